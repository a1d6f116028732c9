"""Pins for the float64 oracle (CPU only).

The oracle is trusted only because these tests tie it to things other than
itself: analytic fixtures (tests/golden), PyTorch's own float64
scaled_dot_product_attention and logsumexp, closed forms (Q=0, constant V,
causal row 0, a single key, rows summing to 1) and structural invariants
(layout swap, key permutation, GQA == repeated heads, paged == contiguous,
decode == a one-row prefill, extend == per-sequence prefill against the
gathered pages, and a pure-Python brute force of extend).  ``test_mutants_are_caught`` plants plausible
mistakes in a copy of the oracle's C source and checks the pins fail.
"""
import glob
import json
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = 1e-12


def _sdpa_ref(q, k, v, scale, mask=None):
    """PyTorch float64 SDPA on [B,H,S,D] tensors; ``mask`` is a bool [S_q,S_kv]."""
    return F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)


def _lse_ref(q, k, scale, mask=None):
    s = scale * torch.matmul(q, k.transpose(-1, -2))
    if mask is not None:
        s = s.masked_fill(~mask, float("-inf"))
    return torch.logsumexp(s, dim=-1)


def _bottom_right(S_q, S_kv):
    return torch.ones(S_q, S_kv, dtype=torch.bool).tril(diagonal=S_kv - S_q)


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64)


# ------------------------------------------------------------------ golden


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(GOLDEN, "*.json"))),
                         ids=lambda p: os.path.basename(p))
def test_golden_fixture(path):
    with open(path) as f:
        fx = json.load(f)
    if fx["kind"] == "prefill":
        layout = oracle.BHSD if fx["layout"] == "bhsd" else oracle.BSHD
        o, lse = oracle.prefill(np.array(fx["q"]), np.array(fx["k"]), np.array(fx["v"]),
                                causal=fx["causal"], scale=fx["scale"], layout=layout,
                                n_threads=2)
    else:
        o, lse = oracle.decode(np.array(fx["q"]), np.array(fx["k_pool"]),
                               np.array(fx["v_pool"]), np.array(fx["kv_lens"]),
                               scale=fx["scale"], page_table=np.array(fx["page_table"]),
                               n_threads=2)
    np.testing.assert_allclose(o, np.array(fx["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(fx["lse"]), rtol=0, atol=1e-12)


# ------------------------------------------------------- library routines


@pytest.mark.parametrize("B,H,S_q,S_kv,D", [(1, 1, 1, 1, 8), (2, 3, 17, 17, 8),
                                            (1, 2, 33, 70, 64), (2, 1, 64, 64, 128)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
def test_prefill_matches_torch_sdpa(B, H, S_q, S_kv, D, causal, layout):
    q = _rand((B, H, S_q, D), 1)
    k = _rand((B, H, S_kv, D), 2)
    v = _rand((B, H, S_kv, D), 3)
    scale = 1.0 / math.sqrt(D)
    mask = _bottom_right(S_q, S_kv) if causal else None
    ref_o = _sdpa_ref(q, k, v, scale, mask)
    ref_lse = _lse_ref(q, k, scale, mask)
    if layout == "bhsd":
        o, lse = oracle.prefill(q, k, v, causal=causal, scale=scale, layout=oracle.BHSD)
        o = torch.from_numpy(o)
    else:
        t = lambda x: x.transpose(1, 2).contiguous()  # noqa: E731
        o, lse = oracle.prefill(t(q), t(k), t(v), causal=causal, scale=scale,
                                layout=oracle.BSHD)
        o = torch.from_numpy(o).transpose(1, 2)
    torch.testing.assert_close(o, ref_o, rtol=0, atol=TOL)
    torch.testing.assert_close(torch.from_numpy(lse), ref_lse, rtol=0, atol=TOL)


def test_causal_square_matches_torch_is_causal():
    """With S_q == S_kv the bottom-right mask is PyTorch's top-left is_causal."""
    q, k, v = _rand((1, 2, 40, 16), 4), _rand((1, 2, 40, 16), 5), _rand((1, 2, 40, 16), 6)
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=0.3)
    o, _ = oracle.prefill(q, k, v, causal=True, scale=0.3)
    torch.testing.assert_close(torch.from_numpy(o), ref, rtol=0, atol=TOL)


def test_bottom_right_is_tail_of_square():
    """Causal rows with S_q < S_kv equal the last S_q rows of the square problem."""
    S_kv, S_q = 50, 13
    q_full, k, v = _rand((1, 1, S_kv, 16), 7), _rand((1, 1, S_kv, 16), 8), _rand((1, 1, S_kv, 16), 9)
    o_full, lse_full = oracle.prefill(q_full, k, v, causal=True, scale=0.25)
    o_tail, lse_tail = oracle.prefill(q_full[:, :, -S_q:], k, v, causal=True, scale=0.25)
    np.testing.assert_allclose(o_tail, o_full[:, :, -S_q:], rtol=0, atol=TOL)
    np.testing.assert_allclose(lse_tail, lse_full[:, :, -S_q:], rtol=0, atol=TOL)


# ------------------------------------------------------------ closed forms


@pytest.mark.parametrize("causal", [False, True])
def test_zero_q_gives_mean_of_visible_v(causal):
    S_q, S_kv, D = 9, 21, 8
    q = torch.zeros(1, 1, S_q, D, dtype=torch.float64)
    k, v = _rand((1, 1, S_kv, D), 10), _rand((1, 1, S_kv, D), 11)
    o, lse = oracle.prefill(q, k, v, causal=causal, scale=0.5)
    for i in range(S_q):
        n_vis = min(S_kv, i + S_kv - S_q + 1) if causal else S_kv
        mean = v[0, 0, :n_vis].mean(dim=0).numpy()
        np.testing.assert_allclose(o[0, 0, i], mean, rtol=0, atol=TOL)
        assert abs(lse[0, 0, i] - math.log(n_vis)) < TOL


def test_zero_k_gives_uniform_weights():
    q, v = _rand((1, 1, 5, 8), 12), _rand((1, 1, 7, 8), 13)
    k = torch.zeros(1, 1, 7, 8, dtype=torch.float64)
    o, lse = oracle.prefill(q, k, v, causal=False, scale=0.5)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0].mean(0).numpy(), (5, 8)),
                               rtol=0, atol=TOL)
    np.testing.assert_allclose(lse, math.log(7), rtol=0, atol=TOL)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_constant_o(causal):
    q, k = _rand((2, 2, 11, 8), 14), _rand((2, 2, 11, 8), 15)
    v = torch.full((2, 2, 11, 8), -3.25, dtype=torch.float64)
    o, _ = oracle.prefill(q, k, v, causal=causal, scale=1.0)
    np.testing.assert_allclose(o, -3.25, rtol=0, atol=TOL)


def test_causal_row_zero_is_v0():
    q, k, v = _rand((1, 3, 12, 16), 16), _rand((1, 3, 12, 16), 17), _rand((1, 3, 12, 16), 18)
    o, lse = oracle.prefill(q, k, v, causal=True, scale=0.7)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0].numpy(), rtol=0, atol=TOL)
    expect = 0.7 * (q[:, :, 0] * k[:, :, 0]).sum(-1)
    np.testing.assert_allclose(lse[:, :, 0], expect.numpy(), rtol=0, atol=TOL)


def test_single_key_gives_its_value():
    q, k, v = _rand((2, 2, 6, 8), 19), _rand((2, 2, 1, 8), 20), _rand((2, 2, 1, 8), 21)
    o, _ = oracle.prefill(q, k, v, causal=False, scale=0.9)
    np.testing.assert_allclose(o, np.broadcast_to(v.numpy(), o.shape), rtol=0, atol=TOL)


def test_rows_sum_to_one():
    """With V = identity (D = S_kv) each output row is the softmax row itself."""
    S = 24
    q, k = _rand((1, 1, S, S), 22), _rand((1, 1, S, S), 23)
    v = torch.eye(S, dtype=torch.float64).view(1, 1, S, S)
    for causal in (False, True):
        o, _ = oracle.prefill(q, k, v, causal=causal, scale=0.4)
        np.testing.assert_allclose(o.sum(-1), 1.0, rtol=0, atol=TOL)
        assert (o >= 0).all()
        if causal:  # nothing leaks to future keys
            assert np.abs(np.triu(o[0, 0], k=1)).max() == 0.0


def test_key_permutation_invariance():
    q, k, v = _rand((1, 2, 8, 16), 24), _rand((1, 2, 30, 16), 25), _rand((1, 2, 30, 16), 26)
    perm = torch.randperm(30, generator=torch.Generator().manual_seed(0))
    o1, l1 = oracle.prefill(q, k, v, causal=False, scale=0.3)
    o2, l2 = oracle.prefill(q, k[:, :, perm], v[:, :, perm], causal=False, scale=0.3)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=TOL)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=TOL)


def test_fully_masked_rows_and_empty_kv():
    q, k, v = _rand((1, 1, 6, 8), 27), _rand((1, 1, 4, 8), 28), _rand((1, 1, 4, 8), 29)
    # S_q > S_kv, causal: rows 0 and 1 see no key (i + S_kv - S_q < 0)
    o, lse = oracle.prefill(q, k, v, causal=True, scale=0.5)
    assert np.all(o[0, 0, :2] == 0.0) and np.all(np.isneginf(lse[0, 0, :2]))
    assert np.all(np.isfinite(lse[0, 0, 2:]))
    np.testing.assert_allclose(o[0, 0, 2], v[0, 0, 0].numpy(), rtol=0, atol=TOL)
    o, lse = oracle.prefill(q, k[:, :, :0], v[:, :, :0], causal=False, scale=0.5)
    assert np.all(o == 0.0) and np.all(np.isneginf(lse))


# ------------------------------------------------------------------ decode


def _decode_torch_ref(inp, scale):
    """Per sequence: PyTorch SDPA over its first kv_len contiguous keys, GQA by
    repeat_interleave of the kv heads."""
    cont = workloads.contiguous_view_of(inp)
    B, H_q, D = cont.q.shape
    H_kv = cont.k.shape[2]
    outs, lses = [], []
    for b in range(B):
        n = int(cont.kv_lens[b])
        qb = cont.q[b].double().view(1, H_q, 1, D)
        kb = cont.k[b, :n].double().permute(1, 0, 2).repeat_interleave(H_q // H_kv, 0)[None]
        vb = cont.v[b, :n].double().permute(1, 0, 2).repeat_interleave(H_q // H_kv, 0)[None]
        outs.append(F.scaled_dot_product_attention(qb, kb, vb, scale=scale)[0, :, 0])
        lses.append(_lse_ref(qb, kb, scale)[0, :, 0])
    return torch.stack(outs), torch.stack(lses)


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("H_q,H_kv", [(4, 4), (8, 2), (6, 1)])
def test_decode_matches_torch_sdpa(paged, H_q, H_kv):
    case = workloads.DecodeCase("t", 3, H_q, H_kv, 16, 1, 45, 48, paged=paged, page_size=16,
                                dtype="bf16", seed=3)
    inp = workloads.make_decode(case)
    o, lse = oracle.decode(inp.q, inp.k, inp.v, inp.kv_lens, scale=case.scale,
                           page_table=inp.page_table)
    ref_o, ref_lse = _decode_torch_ref(inp, case.scale)
    torch.testing.assert_close(torch.from_numpy(o), ref_o, rtol=0, atol=TOL)
    torch.testing.assert_close(torch.from_numpy(lse), ref_lse, rtol=0, atol=TOL)


def test_decode_paged_equals_contiguous():
    case = workloads.DecodeCase("t", 4, 8, 2, 32, 1, 70, 80, paged=True, page_size=16, seed=5)
    inp = workloads.make_decode(case)
    cont = workloads.contiguous_view_of(inp)
    o1, l1 = oracle.decode(inp.q, inp.k, inp.v, inp.kv_lens, scale=0.2, page_table=inp.page_table)
    o2, l2 = oracle.decode(cont.q, cont.k, cont.v, cont.kv_lens, scale=0.2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_decode_gqa_equals_repeated_heads():
    case = workloads.DecodeCase("t", 2, 8, 2, 16, 5, 40, 40, paged=False, seed=6)
    inp = workloads.make_decode(case)
    k_rep = inp.k.repeat_interleave(4, dim=2)
    v_rep = inp.v.repeat_interleave(4, dim=2)
    o1, l1 = oracle.decode(inp.q, inp.k, inp.v, inp.kv_lens, scale=0.25)
    o2, l2 = oracle.decode(inp.q, k_rep, v_rep, inp.kv_lens, scale=0.25)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=TOL)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=TOL)


def test_decode_equals_one_row_prefill():
    case = workloads.DecodeCase("t", 2, 4, 4, 16, 3, 30, 30, paged=False, seed=7)
    inp = workloads.make_decode(case)
    o, lse = oracle.decode(inp.q, inp.k, inp.v, inp.kv_lens, scale=0.3)
    for b in range(2):
        n = int(inp.kv_lens[b])
        q = inp.q[b].view(1, 1, 4, 16)  # BSHD with S_q = 1
        po, plse = oracle.prefill(q, inp.k[b:b + 1, :n], inp.v[b:b + 1, :n], causal=False,
                                  scale=0.3, layout=oracle.BSHD)
        np.testing.assert_allclose(o[b], po[0, 0], rtol=0, atol=TOL)
        np.testing.assert_allclose(lse[b], plse[0, :, 0], rtol=0, atol=TOL)


def test_decode_empty_sequence():
    case = workloads.DecodeCase("t", 2, 2, 1, 8, 0, 0, 16, paged=True, page_size=16, seed=8)
    inp = workloads.make_decode(case, kv_lens=[0, 5])
    o, lse = oracle.decode(inp.q, inp.k, inp.v, inp.kv_lens, scale=1.0, page_table=inp.page_table)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(o[1])) and np.all(np.abs(o[1]) < 100)


def test_oracle_rejects_bad_arguments():
    q = np.zeros((1, 3, 4))
    k = np.zeros((1, 4, 2, 4))
    with pytest.raises(RuntimeError):  # H_q % H_kv != 0
        oracle.decode(q, k, k, np.array([2]), scale=1.0)
    with pytest.raises(RuntimeError):  # kv_len beyond the cache
        oracle.decode(np.zeros((1, 2, 4)), k, k, np.array([5]), scale=1.0)


# ------------------------------------------------------------------ extend


def _extend_torch_ref(inp, causal, scale):
    """Per sequence: gather its kv_len keys through the page table with torch
    indexing, repeat kv heads for GQA and call PyTorch float64 SDPA with an
    explicit bottom-right mask."""
    B, S_q, H_q, D = inp.q.shape
    H_kv = inp.k.shape[2]
    ps = inp.page_size
    outs, lses = [], []
    for b in range(B):
        n = int(inp.kv_lens[b])
        t = torch.arange(n)
        phys = inp.page_table[b].long()[t // ps]
        kb = inp.k[phys, t % ps].double().permute(1, 0, 2).repeat_interleave(H_q // H_kv, 0)[None]
        vb = inp.v[phys, t % ps].double().permute(1, 0, 2).repeat_interleave(H_q // H_kv, 0)[None]
        qb = inp.q[b].double().permute(1, 0, 2)[None]  # [1, H_q, S_q, D]
        mask = _bottom_right(S_q, n) if causal else torch.ones(S_q, n, dtype=torch.bool)
        o = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, scale=scale)
        lse = _lse_ref(qb, kb, scale, mask)
        empty = ~mask.any(dim=1)  # rows with no visible key: o = 0 by definition
        o[:, :, empty] = 0.0
        outs.append(o[0].permute(1, 0, 2))
        lses.append(lse[0])
    return torch.stack(outs), torch.stack(lses)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("H_q,H_kv,page_size", [(4, 4, 16), (8, 2, 8), (6, 1, 64)])
def test_extend_matches_torch_sdpa(causal, H_q, H_kv, page_size):
    case = workloads.ExtendCase("t", 3, 21, H_q, H_kv, 16, 0, 60, page_size=page_size,
                                causal=causal, seed=11)
    inp = workloads.make_extend(case)
    o, lse = oracle.extend(inp.q, inp.k, inp.v, inp.page_table, inp.kv_lens, causal=causal,
                           scale=case.scale)
    ref_o, ref_lse = _extend_torch_ref(inp, causal, case.scale)
    torch.testing.assert_close(torch.from_numpy(o), ref_o, rtol=0, atol=TOL)
    torch.testing.assert_close(torch.from_numpy(lse), ref_lse, rtol=0, atol=TOL)


def test_extend_brute_force_tiny():
    """Pure-Python loops over a 2-sequence, 3-query, 8-token-page case."""
    case = workloads.ExtendCase("t", 2, 3, 2, 1, 4, 0, 6, page_size=8, causal=True, seed=12)
    inp = workloads.make_extend(case, prefix_lens=[6, 0])
    scale = 0.7
    o, lse = oracle.extend(inp.q, inp.k, inp.v, inp.page_table, inp.kv_lens, causal=True,
                           scale=scale)
    q = inp.q.double().tolist()
    k = inp.k.double().tolist()
    v = inp.v.double().tolist()
    for b in range(2):
        n = int(inp.kv_lens[b])
        for h in range(2):
            for i in range(3):
                keys = range(0, i + n - 3 + 1)
                s = []
                for j in keys:
                    pg, sl = int(inp.page_table[b, j // 8]), j % 8
                    s.append(scale * sum(q[b][i][h][d] * k[pg][sl][0][d] for d in range(4)))
                w = [math.exp(x) for x in s]
                tot = sum(w)
                for d in range(4):
                    num = sum(w[jj] * v[int(inp.page_table[b, j // 8])][j % 8][0][d]
                              for jj, j in enumerate(keys))
                    assert abs(o[b, i, h, d] - num / tot) < 1e-12
                assert abs(lse[b, h, i] - math.log(tot)) < 1e-12


def test_extend_short_cache_and_constant_v():
    """kv_len < S_q leaves the first rows with no visible key (o = 0, lse =
    -inf); with V constant per kv head every visible row returns that constant."""
    case = workloads.ExtendCase("t", 2, 10, 4, 2, 8, 0, 5, page_size=8, causal=True, seed=13)
    inp = workloads.make_extend(case, prefix_lens=[0, 5])
    inp.kv_lens[0] = 4  # only 4 cached keys for 10 new queries
    inp.v[:] = torch.arange(2, dtype=inp.v.dtype).view(1, 1, 2, 1) + 3.0
    o, lse = oracle.extend(inp.q, inp.k, inp.v, inp.page_table, inp.kv_lens, causal=True,
                           scale=0.4)
    assert np.all(o[0, :6] == 0.0) and np.all(np.isneginf(lse[0, :, :6]))
    assert np.all(np.isfinite(lse[0, :, 6:])) and np.all(np.isfinite(lse[1]))
    want = np.array([3.0, 3.0, 4.0, 4.0]).reshape(1, 4, 1)  # heads 0,1 -> kv 0; 2,3 -> kv 1
    np.testing.assert_allclose(o[0, 6:], np.broadcast_to(want, (4, 4, 8)), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o[1], np.broadcast_to(want, (10, 4, 8)), rtol=0, atol=1e-12)


def test_extend_without_prefix_equals_causal_prefill():
    """With no cached prefix and identity-free random pages, extend is the
    square causal prefill of the gathered sequence (BSHD)."""
    case = workloads.ExtendCase("t", 2, 37, 4, 4, 16, 0, 0, page_size=16, causal=True, seed=14)
    inp = workloads.make_extend(case)
    o, lse = oracle.extend(inp.q, inp.k, inp.v, inp.page_table, inp.kv_lens, causal=True,
                           scale=0.25)
    for b in range(2):
        t = torch.arange(37)
        phys = inp.page_table[b].long()[t // 16]
        kb, vb = inp.k[phys, t % 16][None], inp.v[phys, t % 16][None]
        po, plse = oracle.prefill(inp.q[b:b + 1], kb, vb, causal=True, scale=0.25,
                                  layout=oracle.BSHD)
        np.testing.assert_allclose(o[b], po[0], rtol=0, atol=TOL)
        np.testing.assert_allclose(lse[b], plse[0], rtol=0, atol=TOL)


# -------------------------------------------------------------------- fp8


def test_e4m3_decode_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ours = oracle.decode_e4m3(codes.numpy())
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and int(nan.sum()) == 2  # 0x7f and 0xff
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_e4m3_decode_closed_forms():
    """Values fixed by the format definition: 1 = 0x38, largest 448 = 0x7e,
    smallest subnormal 2^-9 = 0x01, smallest normal 2^-6 = 0x08, -2 = 0xc0."""
    v = oracle.decode_e4m3(np.array([0x38, 0x7E, 0x01, 0x08, 0xC0, 0x00, 0x07, 0x3C],
                                    dtype=np.uint8))
    assert list(v) == [1.0, 448.0, 2.0 ** -9, 2.0 ** -6, -2.0, 0.0, 7 * 2.0 ** -9, 1.5]


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_fp8_matches_torch_sdpa(causal):
    case = workloads.Fp8PrefillCase("t", 2, 3, 40, 75, 32, "bhsd", causal, seed=31)
    q8, k8, v8, dq, dk, dv = workloads.make_prefill_fp8(case)
    o, lse = oracle.prefill_fp8(q8, k8, v8, descale_q=dq, descale_k=dk, descale_v=dv,
                                causal=causal, scale=case.scale)
    Q, K, V = q8.double() * dq, k8.double() * dk, v8.double() * dv
    mask = _bottom_right(40, 75) if causal else None
    torch.testing.assert_close(torch.from_numpy(o), _sdpa_ref(Q, K, V, case.scale, mask),
                               rtol=0, atol=TOL)
    torch.testing.assert_close(torch.from_numpy(lse), _lse_ref(Q, K, case.scale, mask), rtol=0,
                               atol=TOL)


def test_fp8_quantization_is_within_half_a_step():
    """The input recipe: codes * descale reproduce x within half an E4M3 step."""
    x = torch.randn(1000, generator=torch.Generator().manual_seed(3))
    q8, d = workloads.quantize_e4m3(x)
    y = torch.from_numpy(oracle.decode_e4m3(q8)) * d
    rel = ((y - x.double()).abs() / x.double().abs().clamp_min(2.0 ** -6 * d)).max().item()
    assert rel <= 2.0 ** -4 + 1e-12


# --------------------------------------------------------------- backward


def _torch_grads(q, k, v, dout, scale, mask):
    """PyTorch float64 autograd of SDPA on [B,H,S,D] tensors."""
    q, k, v = (t.detach().clone().requires_grad_(True) for t in (q, k, v))
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    o.backward(dout)
    return q.grad, k.grad, v.grad


@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S_q,S_kv", [(17, 17), (9, 30), (40, 25)])
def test_prefill_bwd_matches_torch_autograd(S_q, S_kv, causal, layout):
    B, H, D = 2, 3, 16
    q, k, v, do = (_rand((B, H, S, D), sd) for S, sd in ((S_q, 51), (S_kv, 52), (S_kv, 53),
                                                          (S_q, 54)))
    mask = _bottom_right(S_q, S_kv) if causal else None
    if causal and S_q > S_kv:
        return  # rows with no visible key: PyTorch yields NaN there (covered below)
    ref = _torch_grads(q, k, v, do, 0.3, mask)
    tr = (lambda x: x) if layout == "bhsd" else (lambda x: x.transpose(1, 2).contiguous())
    ours = oracle.prefill_bwd(tr(q), tr(k), tr(v), tr(do), causal=causal, scale=0.3,
                              layout=oracle.BHSD if layout == "bhsd" else oracle.BSHD)
    for a, r in zip(ours, ref):
        torch.testing.assert_close(torch.from_numpy(a), tr(r), rtol=0, atol=TOL)


def test_prefill_bwd_matches_finite_differences():
    """Gradients of L = sum(dout * O) by central differences of the forward
    oracle, on a tiny causal case (independent of the backward formulas)."""
    B, H, S_q, S_kv, D = 1, 2, 3, 5, 3
    q, k, v, do = (_rand((B, H, S, D), sd).numpy() for S, sd in ((S_q, 61), (S_kv, 62),
                                                                  (S_kv, 63), (S_q, 64)))
    dq, dk, dv = oracle.prefill_bwd(q, k, v, do, causal=True, scale=0.7, n_threads=1)

    def loss(q_, k_, v_):
        o, _ = oracle.prefill(q_, k_, v_, causal=True, scale=0.7, n_threads=1)
        return float((o * do).sum())

    eps = 1e-5
    for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = xp, xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=0, atol=1e-8)


def test_prefill_bwd_invariants():
    """dK sums to zero over the keys of a head (the dS rows sum to zero); a
    zero upstream gradient gives zero gradients; rows with no visible key
    (causal, S_q > S_kv) contribute nothing."""
    B, H, S_q, S_kv, D = 2, 2, 12, 7, 8
    q, k, v, do = (_rand((B, H, S, D), sd).numpy() for S, sd in ((S_q, 71), (S_kv, 72),
                                                                  (S_kv, 73), (S_q, 74)))
    dq, dk, dv = oracle.prefill_bwd(q, k, v, do, causal=False, scale=0.4)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    z = oracle.prefill_bwd(q, k, v, np.zeros_like(do), causal=False, scale=0.4)
    assert all(np.all(a == 0.0) for a in z)
    dq, dk, dv = oracle.prefill_bwd(q, k, v, do, causal=True, scale=0.4)
    assert np.all(dq[:, :, :S_q - S_kv] == 0.0)  # rows 0..4 see no key
    do2 = do.copy()
    do2[:, :, :S_q - S_kv] = 123.0  # their upstream gradient must not matter
    dq2, dk2, dv2 = oracle.prefill_bwd(q, k, v, do2, causal=True, scale=0.4)
    np.testing.assert_array_equal(dk, dk2)
    np.testing.assert_array_equal(dv, dv2)


# ------------------------------------------------------------- MQA logits


def _mqa_torch(q8, kv8, kv_scale, w, start, end, clean):
    """PyTorch float64: per-head scores by einsum, ReLU, weighted head sum,
    window mask."""
    q = q8.double()
    k = kv8.double()
    s = torch.einsum("ihd,jd->ihj", q, k) * kv_scale.double()[None, None, :]
    out = (torch.relu(s) * w.double()[:, :, None]).sum(dim=1)
    j = torch.arange(k.shape[0])[None, :]
    inside = (j >= start.long()[:, None].clamp(min=0)) & (j < end.long()[:, None])
    fill = float("-inf") if clean else float("nan")
    return torch.where(inside, out, torch.full_like(out, fill))


@pytest.mark.parametrize("window", ["causal", "cp", "misaligned", "empty", "past_end"])
@pytest.mark.parametrize("clean", [True, False])
def test_mqa_logits_matches_torch(window, clean):
    case = workloads.MqaCase("t", 23, 70, 8, 32, window, clean, seed=91)
    q8, kv8, sc, w, st, en = workloads.make_mqa(case)
    ours = oracle.mqa_logits(oracle.decode_e4m3(q8), oracle.decode_e4m3(kv8), sc, w, st, en,
                             clean_logits=clean)
    ref = _mqa_torch(q8, kv8, sc, w, st, en, clean).numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    np.testing.assert_array_equal(np.isneginf(ours), np.isneginf(ref))
    fin = np.isfinite(ref)
    np.testing.assert_allclose(ours[fin], ref[fin], rtol=1e-12, atol=1e-12)


def test_mqa_logits_closed_forms():
    """Zero weights give 0 inside the window; a head whose query is the
    negated key contributes nothing (ReLU); an empty or past-the-end window
    leaves the row all -inf (clean) or untouched."""
    S_q, S_kv, H, D = 3, 5, 2, 4
    k = np.arange(S_kv * D, dtype=np.float64).reshape(S_kv, D) / 10.0
    q = np.zeros((S_q, H, D))
    q[:, 0, :] = k[1]     # head 0 aligned with key 1
    q[:, 1, :] = -k[1]    # head 1 opposed: ReLU removes it
    sc = np.full(S_kv, 0.5)
    w = np.array([[2.0, 7.0]] * S_q)
    start = np.array([0, 2, 5], dtype=np.int32)
    end = np.array([5, 2, 9], dtype=np.int32)
    out = oracle.mqa_logits(q, k, sc, w, start, end, clean_logits=True)
    assert out[0, 1] == 2.0 * 0.5 * float(k[1] @ k[1])
    assert np.all(np.isneginf(out[1])) and np.all(np.isneginf(out[2]))
    out = oracle.mqa_logits(q, k, sc, np.zeros_like(w), start, end, clean_logits=False,
                            out=np.full((S_q, S_kv), 3.0))
    assert np.all(out[0] == 0.0) and np.all(out[1:] == 3.0)


# --------------------------------------------------------- planted mistakes

_MUTANTS = {
    "causal_off_by_one": ("long lim = i + (J->S_kv - J->S_q);",
                          "long lim = i + (J->S_kv - J->S_q) - 1;"),
    "causal_top_left": ("long lim = i + (J->S_kv - J->S_q);", "long lim = i;"),
    "dropped_scale": ("k_row[d];\n        s_buf[j] = J->scale * dot;",
                      "k_row[d];\n        s_buf[j] = dot;"),
    "extend_dropped_scale": ("k_seq[j * D + d];\n                s_buf[j] = J->scale * dot;",
                             "k_seq[j * D + d];\n                s_buf[j] = dot;"),
    "lse_without_max": ("*lse_out = m + log(l);\n}", "*lse_out = log(l);\n}"),
    "bshd_as_bhsd": ("return (size_t)(((b * S + s) * H + h) * D + d);",
                     "return (size_t)(((b * H + h) * S + s) * D + d);"),
    "gqa_modulo": ("g = h / group;", "g = h % J->H_kv;"),
    "page_slot": ("long slot = t % page_size;", "long slot = t / page_size;"),
    "extend_causal_top_left": ("long lim = i + (kv_len - J->S_q);", "long lim = i;"),
    "extend_gqa_modulo": ("kvh = h / group;", "kvh = h % J->H_kv;"),
    "extend_q_as_bhsd": ("J->q + (size_t)(((b * J->S_q + i) * J->H_q + h) * D)",
                         "J->q + (size_t)(((b * J->H_q + h) * J->S_q + i) * D)"),
    "extend_lse_index": ("J->lse + (size_t)((b * J->H_q + h) * J->S_q + i)",
                         "J->lse + (size_t)((b * J->S_q + i) * J->H_q + h)"),
    "v_from_k": ("o_row[d] += w * v_seq[t * D + d];", "o_row[d] += w * k_seq[t * D + d];"),
    "bwd_dropped_delta": ("const double ds = p[j] * (dp - Di);", "const double ds = p[j] * dp;"),
    "bwd_dk_from_k": ("dk_row[d] += J->scale * ds * q_row[d];",
                      "dk_row[d] += J->scale * ds * k_row[d];"),
    "bwd_dv_from_ds": ("dv_row[d] += p[j] * do_row[d];", "dv_row[d] += ds * do_row[d];"),
    "mqa_no_relu": ("acc += J->w[i * J->H + h] * (s > 0.0 ? s : 0.0);",
                    "acc += J->w[i * J->H + h] * s;"),
    "mqa_window_inclusive": ("if (j < lo || j >= hi) {", "if (j < lo || j > hi) {"),
    "e4m3_bias_8": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3_subnormal_as_normal": ("v = ldexp((double)m / 8.0, -6);",
                                 "v = ldexp(1.0 + (double)m / 8.0, -7);"),
}


def _pins_pass() -> bool:
    """Run a fast subset of the pins against whatever library oracle._lib holds."""
    checks = [
        lambda: test_prefill_matches_torch_sdpa(1, 2, 33, 70, 64, True, "bshd"),
        lambda: test_prefill_matches_torch_sdpa(2, 1, 64, 64, 128, False, "bhsd"),
        lambda: test_decode_matches_torch_sdpa(True, 8, 2),
        lambda: test_extend_matches_torch_sdpa(True, 8, 2, 8),
        lambda: test_e4m3_decode_matches_torch_for_every_code(),
        lambda: test_prefill_bwd_matches_torch_autograd(9, 30, True, "bshd"),
        lambda: test_mqa_logits_matches_torch("misaligned", True),
        lambda: test_mqa_logits_closed_forms(),
    ] + [lambda p=p: test_golden_fixture(p)
         for p in sorted(glob.glob(os.path.join(GOLDEN, "*.json")))]
    for c in checks:
        try:
            c()
        except AssertionError:
            return False
    return True


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_mutants_are_caught(name):
    old, new = _MUTANTS[name]
    with open(oracle._SRC) as f:
        src = f.read()
    assert src.count(old) == 1, "mutation anchor must match exactly once"
    tmp = tempfile.mkdtemp()
    try:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        so = os.path.join(tmp, "libmutant.so")
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", path, "-o", so,
                        "-lm"], check=True)
        saved = oracle._load()
        import ctypes
        mutant = ctypes.CDLL(so)
        mutant.oracle_prefill_f64.argtypes = saved.oracle_prefill_f64.argtypes
        mutant.oracle_prefill_f64.restype = ctypes.c_int
        mutant.oracle_decode_f64.argtypes = saved.oracle_decode_f64.argtypes
        mutant.oracle_decode_f64.restype = ctypes.c_int
        mutant.oracle_extend_f64.argtypes = saved.oracle_extend_f64.argtypes
        mutant.oracle_extend_f64.restype = ctypes.c_int
        mutant.oracle_e4m3_decode.argtypes = saved.oracle_e4m3_decode.argtypes
        mutant.oracle_e4m3_decode.restype = None
        mutant.oracle_prefill_bwd_f64.argtypes = saved.oracle_prefill_bwd_f64.argtypes
        mutant.oracle_prefill_bwd_f64.restype = ctypes.c_int
        mutant.oracle_mqa_logits_f64.argtypes = saved.oracle_mqa_logits_f64.argtypes
        mutant.oracle_mqa_logits_f64.restype = ctypes.c_int
        oracle._lib = mutant
        try:
            assert not _pins_pass(), "pins did not catch planted mistake %r" % name
        finally:
            oracle._lib = saved
        assert _pins_pass()
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
