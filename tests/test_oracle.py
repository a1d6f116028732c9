"""Pins for the float64 oracle (CPU only).

The oracle is trusted only because these tests tie it to things other than
itself: analytic fixtures (tests/golden), PyTorch's own float64
scaled_dot_product_attention and logsumexp, closed forms (Q=0, constant V,
causal row 0, a single key, rows summing to 1) and structural invariants
(layout swap, key permutation, GQA == repeated heads, paged == contiguous,
decode == a one-row prefill).  ``test_mutants_are_caught`` plants plausible
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


# --------------------------------------------------------- planted mistakes

_MUTANTS = {
    "causal_off_by_one": ("long lim = i + (J->S_kv - J->S_q);",
                          "long lim = i + (J->S_kv - J->S_q) - 1;"),
    "causal_top_left": ("long lim = i + (J->S_kv - J->S_q);", "long lim = i;"),
    "dropped_scale": ("s_buf[j] = J->scale * dot;", "s_buf[j] = dot;"),
    "lse_without_max": ("*lse_out = m + log(l);\n}", "*lse_out = log(l);\n}"),
    "bshd_as_bhsd": ("return (size_t)(((b * S + s) * H + h) * D + d);",
                     "return (size_t)(((b * H + h) * S + s) * D + d);"),
    "gqa_modulo": ("g = h / group;", "g = h % J->H_kv;"),
    "page_slot": ("long slot = t % J->page_size;", "long slot = t / J->page_size;"),
    "v_from_k": ("o_row[d] += w * v_seq[t * D + d];", "o_row[d] += w * k_seq[t * D + d];"),
}


def _pins_pass() -> bool:
    """Run a fast subset of the pins against whatever library oracle._lib holds."""
    checks = [
        lambda: test_prefill_matches_torch_sdpa(1, 2, 33, 70, 64, True, "bshd"),
        lambda: test_prefill_matches_torch_sdpa(2, 1, 64, 64, 128, False, "bhsd"),
        lambda: test_decode_matches_torch_sdpa(True, 8, 2),
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
        oracle._lib = mutant
        try:
            assert not _pins_pass(), "pins did not catch planted mistake %r" % name
        finally:
            oracle._lib = saved
        assert _pins_pass()
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
