"""Failure detection on the GPU without a fault: a wait that nothing completes
gives up after its time limit and reports through the device error word, and
the context stays usable afterwards."""
import pytest
import torch

import attention_flash_attn_fwd_gb300 as attn
import workloads

pytestmark = pytest.mark.gpu

TIMEOUT = 1  # error code of a wait that ran past its limit
SITE = 900   # the self-test's wait


def test_bounded_wait_gives_up_and_reports():
    assert attn.attn_device_error() == 0
    attn.attn_selftest_wait_timeout(50_000_000)  # 50 ms
    word = attn.attn_device_error()
    assert word >> 16 == TIMEOUT and word & 0xFFFF == SITE
    assert attn.attn_device_error() == 0  # reading cleared it
    # The context still runs kernels and their results are unaffected.
    case = workloads.PrefillCase("after", 1, 2, 256, 256, 128, "bhsd", "bf16", True, seed=5)
    q, k, v = (t.cuda() for t in workloads.make_prefill(case))
    o1 = attn.prefill(q, k, v, causal=True)
    attn.attn_selftest_wait_timeout(10_000_000)
    o2 = attn.prefill(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert attn.attn_device_error() >> 16 == TIMEOUT
    assert torch.equal(o1, o2)
    assert attn.attn_device_error() == 0
