"""attn_decode_fwd_noalloc against attn_decode_fwd, through the C ABI.

The allocation-free entry point serves callers that cannot let a library call
cudaMalloc: engines whose framework owns all device memory through its own
pool and budget, and serving loops that must not block on the allocator or
meet an out-of-memory error mid-step.  Its split partials live in a fixed
device array inside the library instead of a grown workspace; the checks,
split plan and kernels are the allocating entry point's own.  So these tests
check that it gives the allocating entry point's results bit for bit (and so
within the oracle tolerance the other tests use), on two calls in a row whose
second call reuses the array the first one left behind, and that it refuses
plans that do not fit the array.

The file name makes pytest collect it last, so a failure here never hides the
results of the other GPU tests; it also passes when run alone in a fresh
process (its first call is the one that looks up the array on the device).
"""
import pytest
import torch

import attention_flash_attn_fwd_gb300 as attn
import workloads
from parity import assert_close

pytestmark = pytest.mark.gpu


def _device_inputs(inp):
    return dict(q=inp.q.cuda(), k=inp.k.cuda(), v=inp.v.cuda(), lens=inp.kv_lens.cuda(),
                pt=inp.page_table.cuda() if inp.page_table is not None else None)


def _call(entry, inp, d, num_splits, scale):
    B, H_q, D = inp.q.shape
    H_kv = inp.k.shape[2]
    paged = d["pt"] is not None
    out = torch.empty_like(d["q"])
    st = entry(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
               d["pt"].data_ptr() if paged else None, d["lens"].data_ptr(), out.data_ptr(),
               B, H_q, H_kv, D, inp.page_size, inp.max_pages if paged else 1,
               inp.k.shape[0] if paged else B, num_splits, scale,
               attn.ATTN_BF16 if inp.q.dtype == torch.bfloat16 else attn.ATTN_F16,
               torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, attn.attn_last_error()
    return out


@pytest.mark.parametrize("paged", [True, False])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_noalloc_matches_allocating_decode_on_two_calls(paged, num_splits):
    first = workloads.DecodeCase("noalloc_a", 8, 32, 8, 128, 1, 4000, 4096, paged=paged, seed=21)
    second = workloads.DecodeCase("noalloc_b", 5, 16, 4, 128, 1, 900, 1024, paged=paged, seed=22)
    for case in (first, second):  # two calls in a row, the second over new inputs
        inp = workloads.make_decode(case)
        d = _device_inputs(inp)
        ref = _call(attn.attn_decode_fwd, inp, d, num_splits, case.scale)
        got = _call(attn.attn_decode_fwd_noalloc, inp, d, num_splits, case.scale)
        torch.cuda.synchronize()
        assert attn.attn_device_error() == 0
        assert_close(got.cpu(), ref.double().cpu(), "noalloc vs decode (%s)" % case.name)
        # Same checks, plan and kernels: any difference would be stale scratch.
        assert torch.equal(got, ref), "noalloc differs from decode (%s)" % case.name


def test_noalloc_rejects_plans_larger_than_its_array():
    # 32 x 32 heads x 64 splits x (128 + 1) floats = 33.8 MB > 16 MiB.
    case = workloads.DecodeCase("noalloc_big", 32, 32, 8, 128, 1, 64, 4096, paged=False, seed=23)
    inp = workloads.make_decode(case)
    d = _device_inputs(inp)
    out = torch.zeros_like(d["q"])
    st = attn.attn_decode_fwd_noalloc(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                                      None, d["lens"].data_ptr(), out.data_ptr(), 32, 32, 8, 128,
                                      4096, 1, 32, 64, case.scale, attn.ATTN_BF16,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_ERR_UNSUPPORTED
    assert "scratch" in attn.attn_last_error()
    torch.cuda.synchronize()
    assert torch.all(out == 0)  # nothing was launched
