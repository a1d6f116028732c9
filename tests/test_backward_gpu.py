"""Attention backward (dQ, dK, dV) parity against the float64 oracle, through
the C ABI.  The forward's o and lse come from the library's own forward."""
import pytest
import torch

import attention_flash_attn_fwd_gb300 as attn
import oracle
import workloads
from parity import assert_close

pytestmark = pytest.mark.gpu


def _run(case):
    q, k, v, do = workloads.make_prefill_bwd(case)
    qc, kc, vc, dc = (t.cuda() for t in (q, k, v, do))
    o, lse = attn.prefill(qc, kc, vc, causal=case.causal, scale=case.scale, layout=case.layout,
                          return_lse=True)
    dq, dk, dv = attn.prefill_bwd(qc, kc, vc, o, dc, lse, causal=case.causal, scale=case.scale,
                                  layout=case.layout)
    torch.cuda.synchronize()
    assert attn.attn_device_error() == 0
    return (q, k, v, do), (dq.cpu(), dk.cpu(), dv.cpu())


def _ref(inputs, case):
    q, k, v, do = inputs
    return oracle.prefill_bwd(q, k, v, do, causal=case.causal, scale=case.scale,
                              layout=oracle.BHSD if case.layout == "bhsd" else oracle.BSHD)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,S_q,S_kv", [(1, 2, 128, 128), (2, 2, 200, 333), (1, 2, 333, 200),
                                          (1, 1, 65, 700), (1, 1, 1, 130)])
def test_backward_matches_oracle(B, H, S_q, S_kv, causal, layout, dtype):
    case = workloads.PrefillCase("t", B, H, S_q, S_kv, 128, layout, dtype, causal, seed=81)
    inputs, grads = _run(case)
    for name, g, r in zip(("dq", "dk", "dv"), grads, _ref(inputs, case)):
        assert_close(g, r, "%s %s" % (name, case))


def test_backward_is_deterministic_and_dk_sums_to_zero():
    """No atomics: two runs give the same bits.  The dS rows sum to zero, so
    dK summed over the keys of a head is ~0 relative to its size."""
    case = workloads.PrefillCase("t", 2, 2, 512, 512, 128, "bhsd", "bf16", False, seed=82)
    _, g1 = _run(case)
    _, g2 = _run(case)
    assert all(torch.equal(a, b) for a, b in zip(g1, g2))
    dk = g1[1].double()
    assert (dk.sum(dim=2).norm() / dk.norm()).item() < 2e-2


@pytest.mark.parametrize("case", [workloads.C8, workloads.C8_CAUSAL], ids=lambda c: c.name)
def test_backward_full_size_sampled_head(case):
    """The measured backward workload at full size, one sampled (b, h) head
    checked in full against the oracle."""
    inputs, grads = _run(case)
    g = torch.Generator().manual_seed(83)
    b = int(torch.randint(case.B, (1,), generator=g))
    h = int(torch.randint(case.H, (1,), generator=g))
    sl = lambda x: x[b:b + 1, h:h + 1]
    sub = workloads.PrefillCase("s", 1, 1, case.S_q, case.S_kv, case.D, case.layout, case.dtype,
                                case.causal)
    refs = oracle.prefill_bwd(*(sl(x) for x in inputs), causal=case.causal, scale=sub.scale)
    for name, gr, r in zip(("dq", "dk", "dv"), grads, refs):
        assert_close(sl(gr), r, "%s %s b=%d h=%d" % (name, case.name, b, h))
