"""Host-side benchmark logic on CPU: the multi-rank time reduction (gloo,
world size 2) and the JSON-facing helpers."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench
import workloads


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.reduce_max(1.5 + rank)  # rank 1 is the slow one
        bench._barrier()
        q.put((rank, got))
    finally:
        torch.distributed.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 2.5, 1: 2.5}


def test_reduce_max_single_process_is_identity():
    assert bench.reduce_max(3.25) == 3.25


def test_rate_units():
    assert bench._rate(2e12, 1000.0, "TFLOP/s") == pytest.approx(2.0)
    assert bench._rate(5e9, 1.0, "GB/s") == pytest.approx(5000.0)


def test_visible_pair_counts():
    assert workloads.visible_pairs(4, 4, False) == 16
    assert workloads.visible_pairs(4, 4, True) == 10
    assert workloads.visible_pairs(2, 5, True) == 4 + 5  # bottom-right alignment
    assert workloads.visible_pairs(5, 2, True) == 0 + 0 + 0 + 1 + 2
    assert workloads.C2_CAUSAL.flops() == pytest.approx(4 * 4 * 32 * 128 * 4096 * 4097 / 2)


def test_clock_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler(0)
    c.lines = ["0, 1800, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 1900, 2070, 950.1, 0x0, Not Active, Not Active, Not Active, Not Active"]
    s = c.summary()
    assert s["sm_mhz"] == 1850 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
