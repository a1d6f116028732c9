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


def errors(out, ref):
    """(max_abs, rel_l2) of a GPU output against a float64 reference."""
    o = out.detach().to("cpu").double() if isinstance(out, torch.Tensor) else torch.as_tensor(out)
    r = torch.as_tensor(np.asarray(ref), dtype=torch.float64)
    d = o.double() - r
    max_abs = d.abs().max().item() if d.numel() else 0.0
    den = r.norm().item()
    rel = d.norm().item() / den if den > 0 else d.norm().item()
    return max_abs, rel


def assert_close(out, ref, what=""):
    max_abs, rel = errors(out, ref)
    assert max_abs <= MAX_ABS and rel <= REL_L2, (
        "%s: max_abs=%.3e (<= %.0e) rel_l2=%.3e (<= %.0e)" % (what, max_abs, MAX_ABS, rel, REL_L2))
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
