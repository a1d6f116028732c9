"""Prefill kernel parity against the float64 oracle, through the C ABI."""
import math

import pytest
import torch

import attention_flash_attn_fwd_gb300 as attn
import oracle
import workloads
from parity import assert_close, assert_lse_close

pytestmark = pytest.mark.gpu

LAYOUT = {"bhsd": oracle.BHSD, "bshd": oracle.BSHD}


def _run(case: workloads.PrefillCase):
    q, k, v = workloads.make_prefill(case)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = attn.prefill(qd, kd, vd, causal=case.causal, scale=case.scale, layout=case.layout,
                          return_lse=True)
    torch.cuda.synchronize()
    assert attn.attn_device_error() == 0
    return (q, k, v), o, lse


def _check_full(case):
    (q, k, v), o, lse = _run(case)
    ref_o, ref_lse = oracle.prefill(q, k, v, causal=case.causal, scale=case.scale,
                                    layout=LAYOUT[case.layout])
    assert_close(o, ref_o, case.name)
    assert_lse_close(lse, ref_lse, case.name)
    return o, lse


def test_tiny_config_matches_oracle():
    """B=1, H=2, S=128, D=64, BHSD fp16, non-causal, scale 1/8, seed 0."""
    _check_full(workloads.C1)


_SHAPES = [  # (B, H, S_q, S_kv): ragged tails, several CTAs, S_q != S_kv
    (1, 2, 300, 300),
    (2, 3, 513, 513),
    (1, 2, 100, 700),
    (1, 1, 700, 260),
    (1, 1, 1, 1),
    (1, 2, 129, 1000),
]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", _SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_prefill_sweep_matches_oracle(shape, causal, layout, dtype, D):
    B, H, S_q, S_kv = shape
    case = workloads.PrefillCase("sweep", B, H, S_q, S_kv, D, layout, dtype, causal, seed=11)
    _check_full(case)


@pytest.mark.parametrize("D,dtype,layout", [(128, "bf16", "bshd"), (64, "fp16", "bhsd")])
def test_persistent_runs_of_units_without_keys(D, dtype, layout):
    """Causal with far fewer keys than queries (bottom-right alignment) over
    more units than SMs: rows before S_q - S_kv see no key, so six of a head's
    eight units have no key in either tile, one has none in its first tile
    only (the diagonal offset 1674 falls inside its second tile), and the
    persistent CTAs take such units back to back.  Those rows are exact zeros
    with lse = -inf; the rest matches the oracle."""
    S_q, S_kv = 2048, 374
    case = workloads.PrefillCase("nokeys", 2, 80, S_q, S_kv, D, layout, dtype, True, seed=13)
    o, lse = _check_full(case)
    dead = S_q - S_kv
    o_dead = o[:, :dead] if layout == "bshd" else o[:, :, :dead]
    assert torch.all(o_dead == 0)
    assert torch.all(torch.isneginf(lse[:, :, :dead]))


def test_empty_kv_gives_zero_and_neg_inf_lse():
    q = torch.randn(1, 2, 40, 64, dtype=torch.float16, device="cuda")
    k = torch.empty(1, 2, 0, 64, dtype=torch.float16, device="cuda")
    o, lse = attn.prefill(q, k, k, return_lse=True)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_constant_v_and_causal_row_zero():
    g = torch.Generator().manual_seed(5)
    q = torch.randn(2, 4, 384, 128, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(2, 4, 384, 128, generator=g).to(torch.bfloat16).cuda()
    v = torch.full((2, 4, 384, 128), 0.75, dtype=torch.bfloat16, device="cuda")
    o = attn.prefill(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert (o.float() - 0.75).abs().max().item() <= 4e-3
    v2 = torch.randn(2, 4, 384, 128, generator=g).to(torch.bfloat16).cuda()
    o2 = attn.prefill(q, k, v2, causal=True)
    torch.cuda.synchronize()
    # Row 0 sees only key 0: its weight is exactly 1, so O[0] == V[0] bit for bit.
    assert torch.equal(o2[:, :, 0], v2[:, :, 0])


def test_zero_q_gives_mean_of_visible_v():
    g = torch.Generator().manual_seed(6)
    S = 260
    k = torch.randn(1, 2, S, 64, generator=g).to(torch.float16)
    v = torch.randn(1, 2, S, 64, generator=g).to(torch.float16)
    q = torch.zeros(1, 2, S, 64, dtype=torch.float16)
    o, lse = attn.prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, return_lse=True)
    torch.cuda.synchronize()
    counts = torch.arange(1, S + 1, dtype=torch.float64)
    mean = v.double().cumsum(dim=2) / counts.view(1, 1, S, 1)
    assert_close(o, mean, "zero-q causal mean")
    assert_lse_close(lse, torch.log(counts).view(1, 1, S).expand(1, 2, S), "zero-q lse")


def test_prefill_is_deterministic():
    case = workloads.PrefillCase("det", 2, 4, 640, 640, 128, "bhsd", "bf16", True, seed=3)
    q, k, v = (t.cuda() for t in workloads.make_prefill(case))
    o1 = attn.prefill(q, k, v, causal=True)
    o2 = attn.prefill(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_persistent_and_per_unit_grids_agree_bitwise():
    """Eager calls run persistent CTAs fed by the stream's unit counter; a
    graph captured on a stream that never ran a prefill has no counter and
    runs one CTA per unit.  Each unit is computed the same way either way."""
    case = workloads.PrefillCase("grid", 3, 5, 777, 901, 128, "bshd", "bf16", True, seed=6)
    q, k, v = (t.cuda() for t in workloads.make_prefill(case))
    o_eager = attn.prefill(q, k, v, causal=True, layout="bshd")
    out = torch.empty_like(o_eager)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        attn.prefill(q, k, v, causal=True, layout="bshd", out=out)
    g.replay()
    torch.cuda.synchronize()
    assert attn.attn_device_error() == 0
    assert torch.equal(o_eager, out)


def test_concurrent_streams_use_their_own_unit_counters():
    """Calls on two streams may overlap on the GPU: each stream's persistent
    CTAs draw from that stream's counter, so both results are complete."""
    cases = [workloads.PrefillCase("s%d" % n, 2, 8, 1024, 1024, 128, "bhsd", "fp16", n == 1,
                                   seed=20 + n) for n in range(2)]
    inputs = [tuple(t.cuda() for t in workloads.make_prefill(c)) for c in cases]
    ref = [attn.prefill(*x, causal=c.causal) for x, c in zip(inputs, cases)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in cases]
    outs = [torch.empty_like(r) for r in ref]
    for _ in range(3):
        for st, x, c, o in zip(streams, inputs, cases, outs):
            with torch.cuda.stream(st):
                attn.prefill(*x, causal=c.causal, out=o)
    torch.cuda.synchronize()
    assert attn.attn_device_error() == 0
    for o, r in zip(outs, ref):
        assert torch.equal(o, r)


def test_output_only_16_byte_aligned():
    """An output 16 bytes into its allocation (16- but not 32-byte aligned)
    is written with 16-byte stores and matches the aligned result."""
    case = workloads.PrefillCase("al", 2, 3, 300, 300, 128, "bhsd", "bf16", True, seed=7)
    q, k, v = (t.cuda() for t in workloads.make_prefill(case))
    ref = attn.prefill(q, k, v, causal=True)
    flat = torch.empty(ref.numel() + 8, device="cuda", dtype=ref.dtype)
    out = flat[8:].view(ref.shape)
    assert out.data_ptr() % 32 == 16
    attn.prefill(q, k, v, causal=True, out=out)
    torch.cuda.synchronize()
    assert attn.attn_device_error() == 0
    assert torch.equal(out, ref)


def test_layouts_agree_bitwise():
    case = workloads.PrefillCase("lay", 2, 3, 333, 333, 128, "bhsd", "fp16", True, seed=4)
    q, k, v = (t.cuda() for t in workloads.make_prefill(case))
    o1 = attn.prefill(q, k, v, causal=True, layout="bhsd")
    t = lambda x: x.transpose(1, 2).contiguous()  # noqa: E731
    o2 = attn.prefill(t(q), t(k), t(v), causal=True, layout="bshd")
    torch.cuda.synchronize()
    assert torch.equal(o1, o2.transpose(1, 2))


# ------------------------------------------------------------ full size
# The measured workloads, compared with the oracle over every output element
# (no sampling).  Each launch runs persistent CTAs that take many units each
# (C2: 2048 units, C3: 2560 units on 152 SMs), so the unit hand-over path (Q
# refill, a K/V ring that continues across units, the O hand-off) is checked
# on every head.  The oracle takes tens of seconds on the host cores here.


def test_full_size_bhsd_fp16_noncausal():
    _check_full(workloads.C2)


def test_full_size_bhsd_fp16_causal():
    _check_full(workloads.C2_CAUSAL)


def test_full_size_bshd_bf16_causal():
    _check_full(workloads.C3)
