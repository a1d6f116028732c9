"""Every form replayed from a CUDA graph gives the bits of an eager call.

The benchmark times each form this way: one eager call on a side stream (it
creates the per-stream state: the prefill unit counter, the decode split
workspace), then a graph captured on that stream and replayed.  Under
capture the prefill counter is reset by a memset node and the persistent CTAs
run as they do eagerly; decode plans its splits on the device.  Each kernel is
deterministic, so the replay must equal the eager result bit for bit.
"""
import pytest
import torch

import attention_flash_attn_fwd_gb300 as attn
import workloads

pytestmark = pytest.mark.gpu


def _graph_equals_eager(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        eager = [t.clone() for t in fn()]
    side.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        static = fn()
    for _ in range(2):  # a second replay finds the counter reset again
        g.replay()
    torch.cuda.synchronize()
    assert attn.attn_device_error() == 0
    assert len(eager) == len(static)
    for a, b in zip(eager, static):
        assert torch.equal(a, b)


@pytest.mark.parametrize("layout,dtype,causal,D", [("bhsd", "fp16", False, 128),
                                                   ("bshd", "bf16", True, 128),
                                                   ("bhsd", "bf16", True, 64)])
def test_prefill_graph_replay(layout, dtype, causal, D):
    # 4 x 20 heads x 5 blocks of 256 rows = 400 units: several per persistent CTA.
    case = workloads.PrefillCase("g", 4, 20, 1100, 1100, D, layout, dtype, causal, seed=51)
    q, k, v = (t.cuda() for t in workloads.make_prefill(case))
    _graph_equals_eager(lambda: attn.prefill(q, k, v, causal=causal, layout=layout,
                                             return_lse=True))


@pytest.mark.parametrize("paged", [False, True])
def test_decode_graph_replay(paged):
    case = workloads.DecodeCase("g", 6, 32, 8, 128, 1, 5000, 5000, paged, seed=52)
    inp = workloads.make_decode(case, kv_lens=[1, 17, 700, 5000, 0, 2049])
    q, k, v, lens = inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.kv_lens.cuda()
    pt = inp.page_table.cuda() if inp.page_table is not None else None
    _graph_equals_eager(lambda: (attn.decode(q, k, v, lens, page_table=pt),))


def test_extend_graph_replay():
    case = workloads.ExtendCase("g", 3, 300, 8, 2, 128, 0, 900, page_size=16, seed=53)
    inp = workloads.make_extend(case, prefix_lens=[0, 37, 900])
    q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
    pt, lens = inp.page_table.cuda(), inp.kv_lens.cuda()
    _graph_equals_eager(lambda: attn.extend(q, k, v, pt, lens, causal=True, return_lse=True))


def test_prefill_fp8_graph_replay():
    case = workloads.Fp8PrefillCase("g", 2, 8, 700, 900, 128, "bshd", True, seed=54)
    q8, k8, v8, dq, dk, dv = workloads.make_prefill_fp8(case)
    q8, k8, v8 = q8.cuda(), k8.cuda(), v8.cuda()
    _graph_equals_eager(lambda: attn.prefill_fp8(q8, k8, v8, descale_q=dq, descale_k=dk,
                                                 descale_v=dv, causal=True, layout="bshd",
                                                 return_lse=True))


def test_backward_graph_replay():
    case = workloads.PrefillCase("g", 2, 4, 640, 640, 128, "bhsd", "bf16", True, seed=55)
    q, k, v, do = (t.cuda() for t in workloads.make_prefill_bwd(case))
    o, lse = attn.prefill(q, k, v, causal=True, return_lse=True)
    torch.cuda.synchronize()
    _graph_equals_eager(lambda: attn.prefill_bwd(q, k, v, o, do, lse, causal=True))


def test_mqa_logits_graph_replay():
    case = workloads.MqaCase("g", 300, 2000, 64, 128, "misaligned", True, seed=56)
    q8, kv8, sc, w, st, en = (t.cuda() for t in workloads.make_mqa(case))
    _graph_equals_eager(lambda: (attn.mqa_logits_fp8(q8, kv8, sc, w, st, en,
                                                     clean_logits=True),))


def test_decode_graph_survives_workspace_growth():
    """A decode call that has to grow its stream's workspace retires the old
    buffer instead of freeing it, so a graph captured before the growth still
    replays into valid memory and gives its eager bits."""
    small = workloads.DecodeCase("g", 2, 8, 2, 128, 300, 600, 640, True, seed=57)
    big = workloads.DecodeCase("g", 16, 32, 8, 128, 9000, 16000, 16384, True, seed=58)
    s_in, b_in = workloads.make_decode(small), workloads.make_decode(big)
    sd = [t.cuda() for t in (s_in.q, s_in.k, s_in.v, s_in.kv_lens, s_in.page_table)]
    bd = [t.cuda() for t in (b_in.q, b_in.k, b_in.v, b_in.kv_lens, b_in.page_table)]
    # Start from no workspace on any stream (no graph of an earlier test is
    # replayed after this), so the small call sizes it and the big one grows it.
    torch.cuda.synchronize()
    assert attn.attn_release_workspace() == attn.ATTN_OK
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        eager = attn.decode(*sd[:4], page_table=sd[4]).clone()
    side.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        static = attn.decode(*sd[:4], page_table=sd[4])
    with torch.cuda.stream(side):  # needs a larger workspace on the same stream
        big_out = attn.decode(*bd[:4], page_table=bd[4])
    g.replay()
    torch.cuda.synchronize()
    assert attn.attn_device_error() == 0
    assert torch.equal(static, eager)
    assert torch.isfinite(big_out.float()).all()
