"""FP8 MQA logits parity against the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import attention_flash_attn_fwd_gb300 as attn
import oracle
import workloads
from parity import MQA_MAX_ABS_REL_RMS, MQA_REL_L2

pytestmark = pytest.mark.gpu

SENTINEL = 7.25  # entries outside the windows must keep it when clean_logits=0


def _run(case):
    q8, kv8, sc, w, st, en = workloads.make_mqa(case)
    out = torch.full((case.S_q, case.S_kv), SENTINEL, device="cuda", dtype=torch.float32)
    attn.mqa_logits_fp8(q8.cuda(), kv8.cuda(), sc.cuda(), w.cuda(), st.cuda(), en.cuda(),
                        clean_logits=case.clean_logits, out=out)
    torch.cuda.synchronize()
    assert attn.attn_device_error() == 0
    return (q8, kv8, sc, w, st, en), out.cpu().double().numpy()


def _ref(inputs, clean, rows=None):
    q8, kv8, sc, w, st, en = inputs
    if rows is not None:  # index the codes as bytes (float8 CPU indexing is not universal)
        q8, w, st, en = q8.view(torch.uint8)[rows], w[rows], st[rows], en[rows]
    base = np.full((q8.shape[0], kv8.shape[0]), SENTINEL)
    return oracle.mqa_logits(oracle.decode_e4m3(q8), oracle.decode_e4m3(kv8), sc, w, st, en,
                             clean_logits=clean, out=base)


def _check(got, ref, what):
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), "%s: -inf pattern" % what
    fin = np.isfinite(ref)
    assert np.all(np.isfinite(got[fin])), what
    d = got[fin] - ref[fin]
    rms = np.sqrt(np.mean(ref[fin] ** 2)) if fin.any() else 0.0
    if fin.any() and rms > 0:
        rel = np.linalg.norm(d) / np.linalg.norm(ref[fin])
        assert rel <= MQA_REL_L2, "%s: rel_l2=%.3e" % (what, rel)
        assert np.abs(d).max() <= MQA_MAX_ABS_REL_RMS * rms, "%s: max_abs=%.3e rms=%.3e" % (
            what, np.abs(d).max(), rms)


@pytest.mark.parametrize("clean", [True, False])
@pytest.mark.parametrize("window", ["causal", "cp", "misaligned", "empty", "past_end"])
@pytest.mark.parametrize("H", [32, 64, 128])
@pytest.mark.parametrize("S_q,S_kv", [(61, 113), (17, 76), (128, 1024), (1, 300), (257, 700)])
def test_mqa_logits_matches_oracle(S_q, S_kv, H, window, clean):
    case = workloads.MqaCase("t", S_q, S_kv, H, 128, window, clean, seed=101)
    inputs, got = _run(case)
    _check(got, _ref(inputs, clean), "mqa %s" % (case,))


@pytest.mark.parametrize("H", [32, 64, 128])
def test_mqa_logits_special_key_scales(H):
    """Negative, zero and very large (beyond 2^100) per-key scales: every
    scale sign and size the kernel's arithmetic distinguishes, mixed within
    the keys one thread handles."""
    case = workloads.MqaCase("t", 61, 300, H, 128, "misaligned", True, seed=103)
    q8, kv8, sc, w, st, en = workloads.make_mqa(case)
    sc = sc.clone()
    sc[0::7] = -sc[0::7]
    sc[3::11] = 0.0
    sc[5::13] = sc[5::13] * 2.0 ** 110
    sc[6::17] = -sc[6::17] * 2.0 ** 110
    out = torch.full((case.S_q, case.S_kv), SENTINEL, device="cuda", dtype=torch.float32)
    attn.mqa_logits_fp8(q8.cuda(), kv8.cuda(), sc.cuda(), w.cuda(), st.cuda(), en.cuda(),
                        clean_logits=True, out=out)
    torch.cuda.synchronize()
    assert attn.attn_device_error() == 0
    got = out.cpu().double().numpy()
    ref = _ref((q8, kv8, sc, w, st, en), True)
    # Per-key relative check: the huge scales would swamp a global norm.
    fin = np.isfinite(ref)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    for j in range(case.S_kv):
        col = fin[:, j]
        if not col.any():
            continue
        r, g = ref[col, j], got[col, j]
        scale = max(np.sqrt(np.mean(r ** 2)), 1e-30)
        assert np.all(np.isfinite(g)), "key %d" % j
        assert np.abs(g - r).max() <= MQA_MAX_ABS_REL_RMS * scale or np.all(r == 0) and np.all(
            g == 0), "key %d: max_abs=%.3e rms=%.3e" % (j, np.abs(g - r).max(), scale)


def test_mqa_logits_strided_output_and_determinism():
    """A row stride wider than S_kv leaves the padding untouched; two runs
    give the same bits."""
    case = workloads.MqaCase("t", 40, 300, 64, 128, "misaligned", True, seed=102)
    q8, kv8, sc, w, st, en = (t.cuda() for t in workloads.make_mqa(case))
    outs = []
    for _ in range(2):
        buf = torch.full((40, 320), SENTINEL, device="cuda", dtype=torch.float32)
        attn.mqa_logits_fp8(q8, kv8, sc, w, st, en, clean_logits=True, out=buf[:, :300])
        torch.cuda.synchronize()
        outs.append(buf.cpu())
    assert torch.all(outs[0][:, 300:] == SENTINEL)
    assert torch.equal(outs[0], outs[1])


def test_mqa_logits_full_size_sampled_rows():
    """The measured long-context case at full size, checked on sampled rows."""
    case = workloads.C9
    inputs, got = _run(case)
    rows = torch.tensor([0, 1, 517, case.S_q - 1])
    ref = _ref(inputs, case.clean_logits, rows=rows)
    _check(got[rows.numpy()], ref, "C9 sampled rows")
