"""Extend (prefill of new tokens against a paged KV cache) parity against the
float64 oracle, through the C ABI."""
import pytest
import torch

import attention_flash_attn_fwd_gb300 as attn
import oracle
import workloads
from parity import assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


def _gpu(inp: workloads.ExtendInputs, causal, scale, k=None, v=None):
    o, lse = attn.extend(inp.q.cuda(), (inp.k if k is None else k).cuda(),
                         (inp.v if v is None else v).cuda(), inp.page_table.cuda(),
                         inp.kv_lens.cuda(), causal=causal, scale=scale, return_lse=True)
    torch.cuda.synchronize()
    assert attn.attn_device_error() == 0
    return o.cpu(), lse.cpu()


def _ref(inp, causal, scale):
    return oracle.extend(inp.q, inp.k, inp.v, inp.page_table, inp.kv_lens, causal=causal,
                         scale=scale)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S_q,H_q,H_kv", [(300, 8, 2), (128, 4, 4), (17, 16, 1), (513, 4, 1)])
def test_extend_matches_oracle(S_q, H_q, H_kv, D, dtype, causal):
    case = workloads.ExtendCase("t", 3, S_q, H_q, H_kv, D, 0, 700, page_size=16, dtype=dtype,
                                causal=causal, seed=21)
    inp = workloads.make_extend(case, prefix_lens=[0, 37, 700])
    o, lse = _gpu(inp, causal, case.scale)
    ref_o, ref_lse = _ref(inp, causal, case.scale)
    assert_close(o, ref_o, "extend %s" % (case,))
    assert_lse_close(lse, ref_lse, "extend lse %s" % (case,))


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128, 256])
def test_extend_page_sizes(page_size):
    case = workloads.ExtendCase("t", 3, 200, 8, 2, 128, 0, 900, page_size=page_size, seed=22)
    inp = workloads.make_extend(case, prefix_lens=[900, 1, 128])
    o, lse = _gpu(inp, True, case.scale)
    ref_o, ref_lse = _ref(inp, True, case.scale)
    assert_close(o, ref_o, "page_size %d" % page_size)
    assert_lse_close(lse, ref_lse, "page_size %d" % page_size)


@pytest.mark.parametrize("prefix", [0, 1, 15, 16, 17, 127, 128, 129, 255, 256, 1000])
def test_extend_prefix_edges(prefix):
    """The sequence end falls at every position relative to pages and tiles."""
    case = workloads.ExtendCase("t", 2, 100, 4, 2, 128, 0, 1000, seed=23)
    inp = workloads.make_extend(case, prefix_lens=[prefix, 1000 - prefix])
    o, lse = _gpu(inp, True, case.scale)
    ref_o, ref_lse = _ref(inp, True, case.scale)
    assert_close(o, ref_o, "prefix %d" % prefix)
    assert_lse_close(lse, ref_lse, "prefix %d" % prefix)


def test_extend_short_cache_rows_have_no_keys():
    """kv_len < S_q: the first S_q - kv_len rows see no key (o = 0, lse = -inf);
    kv_len = 0 leaves the whole sequence empty."""
    case = workloads.ExtendCase("t", 3, 300, 4, 2, 128, 0, 10, seed=24)
    inp = workloads.make_extend(case, prefix_lens=[0, 10, 0])
    inp.kv_lens[0] = 41
    inp.kv_lens[2] = 0
    o, lse = _gpu(inp, True, case.scale)
    ref_o, ref_lse = _ref(inp, True, case.scale)
    assert torch.all(o[0, :259] == 0) and torch.all(o[2] == 0)
    assert torch.all(torch.isneginf(lse[2]))
    assert_close(o, ref_o, "short cache")
    assert_lse_close(lse, ref_lse, "short cache")


def test_extend_ignores_non_finite_page_tails():
    """Tail slots and unused pages hold NaN: only keys < kv_len may matter."""
    case = workloads.ExtendCase("t", 3, 150, 8, 2, 128, 0, 500, seed=25)
    inp = workloads.make_extend(case, prefix_lens=[3, 250, 499])
    ref_o, ref_lse = _ref(inp, True, case.scale)
    k, v = inp.k.clone(), inp.v.clone()
    poison = torch.tensor(workloads.POISON).to(k.dtype)
    k[k == poison] = float("nan")
    v[v == poison] = float("nan")
    o, lse = _gpu(inp, True, case.scale, k=k, v=v)
    assert torch.isfinite(o.float()).all()
    assert_close(o, ref_o, "poisoned tails")
    assert_lse_close(lse, ref_lse, "poisoned tails")


def test_extend_without_prefix_equals_prefill():
    """No cached prefix and H_q == H_kv: extend over pages is the causal BSHD
    prefill over the same keys gathered contiguously, bit for bit."""
    case = workloads.ExtendCase("t", 2, 700, 4, 4, 128, 0, 0, seed=26)
    inp = workloads.make_extend(case)
    o, lse = _gpu(inp, True, case.scale)
    for b in range(2):
        t = torch.arange(700)
        phys = inp.page_table[b].long()[t // 16]
        k = inp.k[phys, t % 16][None].cuda()
        v = inp.v[phys, t % 16][None].cuda()
        po, plse = attn.prefill(inp.q[b:b + 1].cuda(), k, v, causal=True, layout="bshd",
                                scale=case.scale, return_lse=True)
        torch.cuda.synchronize()
        assert torch.equal(po.cpu()[0], o[b])
        assert torch.equal(plse.cpu()[0], lse[b])


def test_extend_is_deterministic():
    case = workloads.ExtendCase("t", 2, 333, 8, 2, 128, 0, 2000, seed=27)
    inp = workloads.make_extend(case)
    o1, l1 = _gpu(inp, True, case.scale)
    o2, l2 = _gpu(inp, True, case.scale)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_extend_full_size():
    """The measured workload at full size (prefixes up to 15360 tokens, 1024
    new tokens, 16-token pages, CTA pairs), every (sequence, head, row)
    compared with the oracle."""
    case = workloads.C6
    inp = workloads.make_extend(case)
    o, lse = _gpu(inp, case.causal, case.scale)
    ref_o, ref_lse = _ref(inp, case.causal, case.scale)
    assert_close(o, ref_o, "C6")
    assert_lse_close(lse, ref_lse, "C6 lse")


@pytest.mark.parametrize("D", [64, 128])
def test_extend_paired_ctas_match_unpaired(D):
    """With 16-token pages and an even GQA group, CTA pairs share the page
    gather; the same keys laid out in 128-token pages take the unpaired path.
    Both must give the same bits."""
    case = workloads.ExtendCase("t", 3, 333, 8, 2, D, 0, 1500, page_size=16, seed=29)
    inp = workloads.make_extend(case, prefix_lens=[1500, 5, 700])
    o16, l16 = _gpu(inp, True, case.scale)
    B, H_kv = 3, 2
    cap = inp.max_pages * 16
    n128 = -(-cap // 128)
    k128 = torch.zeros(B * n128, 128, H_kv, D, dtype=inp.k.dtype)
    v128 = torch.zeros_like(k128)
    for b in range(B):
        n = int(inp.kv_lens[b])
        t = torch.arange(n)
        phys = inp.page_table[b].long()[t // 16]
        rows = b * n128 * 128 + t
        k128.view(-1, H_kv, D)[rows] = inp.k[phys, t % 16]
        v128.view(-1, H_kv, D)[rows] = inp.v[phys, t % 16]
    pt128 = torch.arange(B * n128, dtype=torch.int32).view(B, n128)
    re = workloads.ExtendInputs(inp.q, k128, v128, inp.kv_lens, pt128, 128, n128)
    o128, l128 = _gpu(re, True, case.scale)
    assert torch.equal(o16, o128) and torch.equal(l16, l128)
