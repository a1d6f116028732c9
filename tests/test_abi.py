"""The C ABI without a GPU: the library builds and loads, exports every
function include/attn_gb300.h declares, and rejects bad arguments on the host
before anything would be launched."""
import ctypes
import os
import re
import subprocess

import pytest

import attention_flash_attn_fwd_gb300 as attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_gb300.h")


def _declared_functions():
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert _declared_functions() == sorted(attn.EXPORTED)


def test_library_loads_and_exports_every_declared_symbol():
    lib = attn.lib()
    for name in _declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", attn.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(attn_\w+)", out))
    assert set(_declared_functions()) <= exported
    assert attn.attn_version().startswith("attn_gb300")


def test_header_compiles_as_plain_c():
    src = '#include "attn_gb300.h"\nint main(void) { return ATTN_OK; }\n'
    r = subprocess.run(["gcc", "-std=c11", "-fsyntax-only", "-x", "c", "-",
                        "-I" + os.path.join(ROOT, "include"), "-I/usr/local/cuda/include"],
                       input=src, text=True, capture_output=True)
    assert r.returncode == 0, r.stderr


def _prefill(**kw):
    a = dict(q=16, k=16, v=16, o=16, lse=None, B=1, H=1, S_q=8, S_kv=8, D=64, layout=0, dtype=0,
             causal=0, scale=0.125, stream=None)
    a.update(kw)
    return attn.attn_prefill_fwd(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(D=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(D=256), attn.ATTN_ERR_UNSUPPORTED),
    (dict(B=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(S_kv=-3), attn.ATTN_ERR_INVALID_ARG),
    (dict(layout=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(dtype=7), attn.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=-1.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(o=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(k=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(q=8), attn.ATTN_ERR_INVALID_ARG),  # not 16-byte aligned
])
def test_prefill_rejects_bad_arguments(kw, code):
    assert _prefill(**kw) == code
    assert attn.attn_last_error()


def test_prefill_empty_problem_is_a_no_op():
    assert _prefill(B=0, q=None, k=None, v=None, o=None) == attn.ATTN_OK
    assert _prefill(S_q=0) == attn.ATTN_OK
    assert _prefill(H=0) == attn.ATTN_OK


def _decode(**kw):
    a = dict(q=16, k_pool=16, v_pool=16, page_table=None, kv_lens=16, o=16, B=2, H_q=8, H_kv=2,
             D=128, page_size=64, max_pages_per_seq=1, num_pages=2, num_splits=0, scale=0.1,
             dtype=1, stream=None)
    a.update(kw)
    return attn.attn_decode_fwd(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(H_kv=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(H_q=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(H_q=64, H_kv=2), attn.ATTN_ERR_UNSUPPORTED),  # group of 32 > 16
    (dict(D=80), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(num_splits=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(page_size=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(num_pages=3), attn.ATTN_ERR_INVALID_ARG),  # contiguous: num_pages must be B
    (dict(page_table=16, page_size=24, max_pages_per_seq=4, num_pages=9),
     attn.ATTN_ERR_UNSUPPORTED),
    (dict(page_table=16, page_size=16, max_pages_per_seq=0, num_pages=9),
     attn.ATTN_ERR_INVALID_ARG),
    (dict(kv_lens=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(o=4), attn.ATTN_ERR_INVALID_ARG),  # misaligned
])
def test_decode_rejects_bad_arguments(kw, code):
    assert _decode(**kw) == code
    assert attn.attn_last_error()


def test_decode_empty_batch_is_a_no_op():
    assert _decode(B=0, num_pages=0) == attn.ATTN_OK


def _mqa(**kw):
    a = dict(q=16, kv=16, kv_scale=16, weights=16, window_start=16, window_end=16, logits=16,
             S_q=4, S_kv=8, H=64, D=128, logits_stride=8, clean_logits=1, stream=None)
    a.update(kw)
    return attn.attn_mqa_logits_fp8(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(H=48), attn.ATTN_ERR_UNSUPPORTED),
    (dict(D=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(S_q=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(logits_stride=7), attn.ATTN_ERR_INVALID_ARG),
    (dict(clean_logits=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(window_end=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(kv=8), attn.ATTN_ERR_INVALID_ARG),  # misaligned
])
def test_mqa_logits_rejects_bad_arguments(kw, code):
    assert _mqa(**kw) == code
    assert attn.attn_last_error()


def test_mqa_logits_empty_problem_is_a_no_op():
    assert _mqa(S_q=0, q=None) == attn.ATTN_OK
    assert _mqa(S_kv=0, logits_stride=0) == attn.ATTN_OK


def _bwd(**kw):
    a = dict(q=16, k=16, v=16, o=16, dout=16, lse=16, dq=16, dk=16, dv=16, delta=16, B=1, H=1,
             S_q=8, S_kv=8, D=128, layout=0, dtype=1, causal=0, scale=0.1, stream=None)
    a.update(kw)
    return attn.attn_prefill_bwd(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(D=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(S_kv=0), attn.ATTN_ERR_UNSUPPORTED),
    (dict(layout=7), attn.ATTN_ERR_INVALID_ARG),
    (dict(dtype=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(causal=5), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=-1.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(delta=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(lse=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(dk=8), attn.ATTN_ERR_INVALID_ARG),  # misaligned
])
def test_backward_rejects_bad_arguments(kw, code):
    assert _bwd(**kw) == code
    assert attn.attn_last_error()


def test_backward_empty_problem_is_a_no_op():
    assert _bwd(B=0, q=None) == attn.ATTN_OK
    assert _bwd(S_q=0, S_kv=0) == attn.ATTN_OK


def _prefill_fp8(**kw):
    a = dict(q=16, k=16, v=16, o=16, lse=None, B=1, H=1, S_q=8, S_kv=8, D=128, layout=0,
             out_dtype=1, causal=0, scale=0.1, descale_q=1.0, descale_k=1.0, descale_v=1.0,
             stream=None)
    a.update(kw)
    return attn.attn_prefill_fp8_fwd(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(D=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(layout=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(out_dtype=4), attn.ATTN_ERR_INVALID_ARG),
    (dict(causal=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(descale_q=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(descale_v=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(descale_k=-2.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(k=4), attn.ATTN_ERR_INVALID_ARG),  # misaligned
])
def test_prefill_fp8_rejects_bad_arguments(kw, code):
    assert _prefill_fp8(**kw) == code
    assert attn.attn_last_error()


def test_prefill_fp8_empty_problem_is_a_no_op():
    assert _prefill_fp8(B=0, q=None, k=None, v=None, o=None) == attn.ATTN_OK
    assert _prefill_fp8(S_q=0) == attn.ATTN_OK


def _extend(**kw):
    a = dict(q=16, k_pool=16, v_pool=16, page_table=16, kv_lens=16, o=16, lse=None, B=2, S_q=64,
             H_q=8, H_kv=2, D=128, page_size=16, max_pages_per_seq=8, num_pages=16, dtype=1,
             causal=1, scale=0.1, stream=None)
    a.update(kw)
    return attn.attn_extend_fwd(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(H_kv=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(H_kv=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(S_q=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=5), attn.ATTN_ERR_INVALID_ARG),
    (dict(causal=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), attn.ATTN_ERR_INVALID_ARG),
    (dict(page_size=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(page_size=4), attn.ATTN_ERR_UNSUPPORTED),
    (dict(page_size=48), attn.ATTN_ERR_UNSUPPORTED),
    (dict(page_size=192), attn.ATTN_ERR_UNSUPPORTED),
    (dict(max_pages_per_seq=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(num_pages=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(page_table=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(kv_lens=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(v_pool=8), attn.ATTN_ERR_INVALID_ARG),  # misaligned
])
def test_extend_rejects_bad_arguments(kw, code):
    assert _extend(**kw) == code
    assert attn.attn_last_error()


def test_extend_empty_problem_is_a_no_op():
    assert _extend(B=0, q=None, o=None) == attn.ATTN_OK
    assert _extend(S_q=0) == attn.ATTN_OK


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "attention_flash_attn_fwd_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, fn)) as f:
                    text = f.read()
                for bad in ("import oracle", "from oracle", "liboracle", "attn_oracle"):
                    assert bad not in text, (fn, bad)


@pytest.mark.parametrize("limit", [0, 10_000_000_001])
def test_selftest_wait_rejects_limits_out_of_range(limit):
    assert attn.lib().attn_selftest_wait_timeout(limit, None) == attn.ATTN_ERR_INVALID_ARG


def test_no_fallback_when_the_library_cannot_be_built():
    """A missing toolkit or library is an error, never a silent host path."""
    code = (
        "import attention_flash_attn_fwd_gb300 as a\n"
        "from attention_flash_attn_fwd_gb300 import _build\n"
        "def no_nvcc(*args, **kw):\n"
        "    raise RuntimeError('nvcc not found')\n"
        "_build.build = no_nvcc\n"
        "try:\n"
        "    a.lib()\n"
        "except RuntimeError as e:\n"
        "    print('raised', e)\n"
        "else:\n"
        "    print('loaded')\n")
    r = subprocess.run(["python", "-c", code], capture_output=True, text=True, cwd=ROOT,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "raised nvcc not found"


@pytest.mark.parametrize("form", ["prefill", "prefill_bwd", "extend", "decode"])
def test_wrappers_reject_host_tensors(form):
    import torch
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensors"):
        if form == "prefill":
            attn.prefill(q, q, q)
        elif form == "prefill_bwd":
            lse = torch.zeros(1, 1, 128, dtype=torch.float32)
            attn.prefill_bwd(q, q, q, q, q, lse)
        elif form == "extend":
            pool = torch.zeros(4, 16, 1, 64, dtype=torch.bfloat16)
            lens = torch.full((1,), 64, dtype=torch.int32)
            table = torch.arange(4, dtype=torch.int32).view(1, 4)
            attn.extend(q.view(1, 128, 1, 64)[:, :16], pool, pool, table, lens)
        else:
            pool = torch.zeros(4, 16, 1, 64, dtype=torch.bfloat16)
            lens = torch.full((1,), 64, dtype=torch.int32)
            table = torch.arange(4, dtype=torch.int32).view(1, 4)
            attn.decode(q.view(1, 128, 64)[:, :1], pool, pool, lens, page_table=table)
