"""Decode (split-KV, paged/contiguous, GQA) parity against the float64 oracle."""
import pytest
import torch

import attention_flash_attn_fwd_gb300 as attn
import oracle
import workloads
from parity import assert_close

pytestmark = pytest.mark.gpu


def _gpu(inp: workloads.DecodeInputs, num_splits=0, scale=None):
    pt = inp.page_table.cuda() if inp.page_table is not None else None
    o = attn.decode(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.kv_lens.cuda(), page_table=pt,
                    num_splits=num_splits, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_device_error() == 0
    return o.cpu()


def _ref(inp, scale):
    o, _ = oracle.decode(inp.q, inp.k, inp.v, inp.kv_lens, scale=scale, page_table=inp.page_table)
    return o


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H_q,H_kv", [(8, 2), (32, 8), (4, 4), (16, 1)])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_decode_matches_oracle(num_splits, H_q, H_kv, D, dtype, paged):
    case = workloads.DecodeCase("t", 4, H_q, H_kv, D, 1, 700, 704, paged=paged, page_size=16,
                                dtype=dtype, seed=2)
    inp = workloads.make_decode(case, kv_lens=[1, 17, 700, 64])
    out = _gpu(inp, num_splits=num_splits, scale=case.scale)
    assert_close(out, _ref(inp, case.scale), "decode %s" % case)


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128])
def test_decode_page_sizes(page_size):
    case = workloads.DecodeCase("t", 3, 8, 2, 128, 1, 1000, 1024, paged=True, page_size=page_size,
                                seed=4)
    inp = workloads.make_decode(case, kv_lens=[1000, 129, 63])
    out = _gpu(inp, scale=case.scale)
    assert_close(out, _ref(inp, case.scale), "page_size %d" % page_size)


@pytest.mark.parametrize("kv", [1, 15, 16, 17, 63, 64, 65, 127, 128, 1000])
def test_decode_length_edges(kv):
    case = workloads.DecodeCase("t", 2, 8, 2, 128, 1, 1024, 1024, paged=True, seed=5)
    inp = workloads.make_decode(case, kv_lens=[kv, 1024 - kv + 1])
    for ns in (0, 2):
        out = _gpu(inp, num_splits=ns, scale=case.scale)
        assert_close(out, _ref(inp, case.scale), "kv=%d splits=%d" % (kv, ns))


def test_decode_zero_length_sequence_gives_zero():
    case = workloads.DecodeCase("t", 3, 8, 2, 128, 0, 0, 256, paged=True, seed=6)
    inp = workloads.make_decode(case, kv_lens=[0, 100, 0])
    out = _gpu(inp, scale=case.scale)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert_close(out, _ref(inp, case.scale), "zero-length")


def test_decode_ignores_non_finite_page_tails():
    """Tail slots and unused pages hold NaN/inf: only keys < kv_len may matter."""
    case = workloads.DecodeCase("t", 3, 8, 2, 128, 1, 500, 512, paged=True, seed=7)
    inp = workloads.make_decode(case, kv_lens=[3, 250, 499])
    ref = _ref(inp, case.scale)
    k, v = inp.k.clone(), inp.v.clone()
    poison = torch.tensor(workloads.POISON).to(k.dtype)
    k[k == poison] = float("nan")
    v[v == poison] = float("inf")
    bad = workloads.DecodeInputs(inp.q, k, v, inp.kv_lens, inp.page_table, inp.page_size,
                                 inp.max_pages)
    out = _gpu(bad, scale=case.scale)
    assert torch.isfinite(out.float()).all()
    assert_close(out, ref, "poisoned tails")
    cont = workloads.contiguous_view_of(inp)
    kc, vc = cont.k.clone(), cont.v.clone()
    kc[kc == poison] = float("nan")
    vc[vc == poison] = float("nan")
    out_c = _gpu(workloads.DecodeInputs(cont.q, kc, vc, cont.kv_lens, None, cont.page_size, 1),
                 scale=case.scale)
    assert_close(out_c, ref, "poisoned contiguous rows")


def test_paged_equals_contiguous_bitwise():
    case = workloads.DecodeCase("t", 5, 32, 8, 128, 1, 3000, 3072, paged=True, seed=8)
    inp = workloads.make_decode(case)
    cont = workloads.contiguous_view_of(inp)
    for ns in (0, 1, 4):
        assert torch.equal(_gpu(inp, num_splits=ns, scale=case.scale),
                           _gpu(cont, num_splits=ns, scale=case.scale))


def test_split_count_does_not_change_result():
    case = workloads.DecodeCase("t", 3, 16, 4, 128, 2000, 6000, 6144, paged=False, seed=9)
    inp = workloads.make_decode(case)
    ref = _ref(inp, case.scale)
    outs = [_gpu(inp, num_splits=ns, scale=case.scale) for ns in (1, 2, 7, 0)]
    for o in outs:
        assert_close(o, ref, "splits")
    for o in outs[1:]:
        assert (o.float() - outs[0].float()).abs().max().item() <= 1e-2


def test_decode_equals_prefill_row():
    """Decode of one query == a one-row (S_q = 1) prefill over the same keys."""
    case = workloads.DecodeCase("t", 1, 8, 8, 128, 777, 777, 777, paged=False, seed=10)
    inp = workloads.make_decode(case)
    out = _gpu(inp, scale=case.scale)
    q = inp.q.view(1, 1, 8, 128).cuda()  # BSHD with S_q = 1
    pre = attn.prefill(q, inp.k.cuda(), inp.v.cuda(), layout="bshd", scale=case.scale)
    torch.cuda.synchronize()
    assert (pre.view(1, 8, 128).cpu().float() - out.float()).abs().max().item() <= 1e-2


def test_decode_is_deterministic():
    case = workloads.DecodeCase("t", 4, 32, 8, 128, 100, 4000, 4096, paged=True, seed=11)
    inp = workloads.make_decode(case)
    assert torch.equal(_gpu(inp, scale=case.scale), _gpu(inp, scale=case.scale))


# ------------------------------------------------------------ full size


@pytest.fixture(scope="module")
def contiguous_full():
    return workloads.make_decode(workloads.C4)


@pytest.fixture(scope="module")
def paged_full():
    return workloads.make_decode(workloads.C5)


def _check_all_sequences(inp, out, scale):
    """Compare every output element with the oracle.  The oracle runs one
    sequence at a time over that sequence's own keys (its pages gathered in
    table order: data movement only) so no call widens the whole pool to
    float64; the per-sequence results fill one reference tensor, compared as
    a whole."""
    ref = torch.empty(out.shape, dtype=torch.float64)
    for b in range(inp.q.shape[0]):
        n = int(inp.kv_lens[b])
        if inp.page_table is None:
            sub = workloads.DecodeInputs(inp.q[b:b + 1], inp.k[b:b + 1, :n], inp.v[b:b + 1, :n],
                                         inp.kv_lens[b:b + 1], None, n, 1)
        else:
            pages = inp.page_table[b, : -(-n // inp.page_size)].long()
            sub = workloads.DecodeInputs(inp.q[b:b + 1], inp.k[pages], inp.v[pages],
                                         inp.kv_lens[b:b + 1],
                                         torch.arange(len(pages), dtype=torch.int32).view(1, -1),
                                         inp.page_size, len(pages))
        ref[b:b + 1] = torch.from_numpy(_ref(sub, scale))
    assert_close(out, ref, "all %d sequences" % inp.q.shape[0])


def test_full_size_contiguous(contiguous_full):
    inp = contiguous_full
    out = _gpu(inp, scale=workloads.C4.scale)
    _check_all_sequences(inp, out, workloads.C4.scale)


def test_full_size_paged(paged_full):
    inp = paged_full
    out = _gpu(inp, scale=workloads.C5.scale)
    _check_all_sequences(inp, out, workloads.C5.scale)


def test_decode_concurrent_streams_do_not_share_partials():
    """Two decode calls on different streams, launched back to back so their
    kernels can overlap: each stream has its own split workspace, so each
    result equals the same call made alone."""
    case = workloads.DecodeCase("t", 8, 32, 8, 128, 2000, 8000, 8192, paged=True, seed=9)
    a = workloads.make_decode(case)
    b = workloads.make_decode(workloads.DecodeCase("t", 8, 32, 8, 128, 2000, 8000, 8192,
                                                   paged=True, seed=10))
    dev = [[t.cuda() for t in (x.q, x.k, x.v, x.kv_lens, x.page_table)] for x in (a, b)]
    alone = []
    for q, k, v, lens, pt in dev:
        alone.append(attn.decode(q, k, v, lens, page_table=pt, scale=case.scale))
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = [torch.empty_like(dev[0][0]), torch.empty_like(dev[1][0])]
    for _ in range(20):
        for (q, k, v, lens, pt), o, s in zip(dev, outs, (s1, s2)):
            with torch.cuda.stream(s):
                attn.decode(q, k, v, lens, page_table=pt, scale=case.scale, out=o)
    torch.cuda.synchronize()
    assert attn.attn_device_error() == 0
    assert torch.equal(outs[0], alone[0]) and torch.equal(outs[1], alone[1])
