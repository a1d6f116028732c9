"""Shared tolerance and error measures for GPU-vs-oracle parity tests.

Tolerance (fp16/bf16 inputs, fp32 accumulation): max-abs error <= 2e-2 and
relative L2 error <= 5e-3 over the whole output tensor; lse (ours) max-abs
<= 1e-3.  Relative L2 = ||O_gpu - O_ref||_2 / ||O_ref||_2.
"""
import numpy as np
import torch

MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_ABS = 1e-3

# FP8 (E4M3) prefill.  The kernel must round P to E4M3 before P V; with 3
# mantissa bits the rounding error of each weight is up to 2^-4 relative
# (rms about 2^-4/sqrt(3) for round-to-nearest), the errors of different keys
# are independent and O = sum_j w_j v_j, so for N(0,1) V the relative L2 error
# of O is about rms(delta) ~ 2-3% at every sequence length (a CPU emulation
# of this rounding gave 1.9-2.7% for S = 128 .. 4096); early causal rows, where
# O is a few V rows of size ~1, reach ~3.5e-2 absolute.  The bounds leave a
# 1.5x / 3x margin.  The scores and lse are not rounded through E4M3.
FP8_MAX_ABS = 1e-1
FP8_REL_L2 = 4e-2

# FP8 MQA logits: E4M3 x E4M3 products are exact and are summed in fp32 (128
# per score by the tensor core, <= 128 heads per logit), so the error is
# ~1e-5 relative; the bounds (relative to the reference's size) leave room
# for a tensor-core accumulator narrower than full fp32.
MQA_REL_L2 = 1e-3
MQA_MAX_ABS_REL_RMS = 1e-2


def errors(out, ref):
    """(max_abs, rel_l2) of a GPU output against a float64 reference."""
    o = out.detach().to("cpu").double() if isinstance(out, torch.Tensor) else torch.as_tensor(out)
    r = torch.as_tensor(np.asarray(ref), dtype=torch.float64)
    d = o.double() - r
    max_abs = d.abs().max().item() if d.numel() else 0.0
    den = r.norm().item()
    rel = d.norm().item() / den if den > 0 else d.norm().item()
    return max_abs, rel


def assert_close(out, ref, what="", max_abs_tol=MAX_ABS, rel_tol=REL_L2):
    max_abs, rel = errors(out, ref)
    assert max_abs <= max_abs_tol and rel <= rel_tol, (
        "%s: max_abs=%.3e (<= %.0e) rel_l2=%.3e (<= %.0e)" % (what, max_abs, max_abs_tol, rel,
                                                              rel_tol))
    return max_abs, rel


def assert_lse_close(lse, ref, what=""):
    l = lse.detach().to("cpu").double()
    r = torch.as_tensor(np.asarray(ref), dtype=torch.float64)
    both_inf = torch.isneginf(l) & torch.isneginf(r)
    assert torch.equal(torch.isneginf(l), torch.isneginf(r)), "%s: -inf rows differ" % what
    d = (l - r).masked_fill(both_inf, 0.0).abs()
    m = d.max().item() if d.numel() else 0.0
    assert m <= LSE_ABS, "%s: lse max_abs=%.3e (<= %.0e)" % (what, m, LSE_ABS)
    return m
