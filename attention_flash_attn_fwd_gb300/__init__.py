"""GB300 (sm_103a) fused attention forward: Python binding of ``libattn_gb300.so``.

The binding only marshals arguments: every step of the computation runs in the
library's CUDA kernels.  There is no CPU or PyTorch fallback; if the library
cannot be built or loaded, importing the functions below raises.

Two layers:

* ``attn_prefill_fwd`` / ``attn_decode_fwd`` -- the C entry points of
  ``include/attn_gb300.h`` with the same names and arguments (raw device
  pointers as ints, ``stream`` as a ``cudaStream_t`` handle int).
* ``prefill`` / ``decode`` -- convenience wrappers over torch CUDA tensors
  (torch is used for device memory and the current stream only).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import _build

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_CUDA = -3
ATTN_ERR_NO_MEMORY = -4
ATTN_ERR_DEVICE_TIMEOUT = -5

ATTN_BHSD = 0
ATTN_BSHD = 1
ATTN_F16 = 0
ATTN_BF16 = 1

_STATUS_NAMES = {
    ATTN_OK: "ATTN_OK",
    ATTN_ERR_INVALID_ARG: "ATTN_ERR_INVALID_ARG",
    ATTN_ERR_UNSUPPORTED: "ATTN_ERR_UNSUPPORTED",
    ATTN_ERR_CUDA: "ATTN_ERR_CUDA",
    ATTN_ERR_NO_MEMORY: "ATTN_ERR_NO_MEMORY",
    ATTN_ERR_DEVICE_TIMEOUT: "ATTN_ERR_DEVICE_TIMEOUT",
}

# Names the header exports (checked against include/attn_gb300.h by the tests).
EXPORTED = ("attn_prefill_fwd", "attn_prefill_bwd", "attn_mqa_logits_fp8", "attn_prefill_fp8_fwd", "attn_extend_fwd", "attn_decode_fwd", "attn_decode_fwd_noalloc",
            "attn_last_error",
            "attn_device_error", "attn_set_wait_limit_ns", "attn_release_workspace",
            "attn_selftest_wait_timeout",
            "attn_version")


class AttnError(RuntimeError):
    """A library call returned a non-OK status."""

    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_STATUS_NAMES.get(status, str(status)), message))
        self.status = status


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the shared library and declare its ABI."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            vp, i32p = ctypes.c_void_p, ctypes.c_void_p
            ci, cf = ctypes.c_int, ctypes.c_float
            L.attn_prefill_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, cf,
                                           vp]
            L.attn_prefill_fwd.restype = ci
            L.attn_mqa_logits_fp8.argtypes = [vp] * 7 + [ci] * 4 + [ctypes.c_int64, ci, vp]
            L.attn_mqa_logits_fp8.restype = ci
            L.attn_prefill_bwd.argtypes = [vp] * 10 + [ci] * 8 + [cf, vp]
            L.attn_prefill_bwd.restype = ci
            L.attn_prefill_fp8_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci,
                                               cf, cf, cf, cf, vp]
            L.attn_prefill_fp8_fwd.restype = ci
            L.attn_extend_fwd.argtypes = [vp, vp, vp, i32p, i32p, vp, vp, ci, ci, ci, ci, ci, ci,
                                          ci, ci, ci, ci, cf, vp]
            L.attn_extend_fwd.restype = ci
            L.attn_decode_fwd.argtypes = [vp, vp, vp, i32p, i32p, vp, ci, ci, ci, ci, ci, ci, ci,
                                          ci, cf, ci, vp]
            L.attn_decode_fwd.restype = ci
            L.attn_decode_fwd_noalloc.argtypes = L.attn_decode_fwd.argtypes
            L.attn_decode_fwd_noalloc.restype = ci
            L.attn_last_error.argtypes = []
            L.attn_last_error.restype = ctypes.c_char_p
            L.attn_device_error.argtypes = [ctypes.POINTER(ctypes.c_int), ci]
            L.attn_device_error.restype = ci
            L.attn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.attn_set_wait_limit_ns.restype = None
            L.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
            L.attn_selftest_wait_timeout.restype = ci
            L.attn_release_workspace.argtypes = []
            L.attn_release_workspace.restype = ci
            L.attn_version.argtypes = []
            L.attn_version.restype = ctypes.c_char_p
            _lib = L
    return _lib


def last_error() -> str:
    return lib().attn_last_error().decode()


def _check(status: int) -> int:
    if status != ATTN_OK:
        raise AttnError(status, last_error())
    return status


# --------------------------------------------------------------- raw C ABI


def attn_prefill_fwd(q, k, v, o, lse, B, H, S_q, S_kv, D, layout, dtype, causal, scale,
                     stream) -> int:
    """C ``attn_prefill_fwd``; pointers and stream as ints.  Returns the status."""
    return lib().attn_prefill_fwd(q, k, v, o, lse, B, H, S_q, S_kv, D, layout, dtype, causal,
                                  scale, stream)


def attn_mqa_logits_fp8(q, kv, kv_scale, weights, window_start, window_end, logits, S_q, S_kv,
                        H, D, logits_stride, clean_logits, stream) -> int:
    """C ``attn_mqa_logits_fp8``; pointers and stream as ints.  Returns the status."""
    return lib().attn_mqa_logits_fp8(q, kv, kv_scale, weights, window_start, window_end, logits,
                                     S_q, S_kv, H, D, logits_stride, clean_logits, stream)


def attn_prefill_bwd(q, k, v, o, dout, lse, dq, dk, dv, delta, B, H, S_q, S_kv, D, layout,
                     dtype, causal, scale, stream) -> int:
    """C ``attn_prefill_bwd``; pointers and stream as ints.  Returns the status."""
    return lib().attn_prefill_bwd(q, k, v, o, dout, lse, dq, dk, dv, delta, B, H, S_q, S_kv, D,
                                  layout, dtype, causal, scale, stream)


def attn_prefill_fp8_fwd(q, k, v, o, lse, B, H, S_q, S_kv, D, layout, out_dtype, causal, scale,
                         descale_q, descale_k, descale_v, stream) -> int:
    """C ``attn_prefill_fp8_fwd``; pointers and stream as ints.  Returns the status."""
    return lib().attn_prefill_fp8_fwd(q, k, v, o, lse, B, H, S_q, S_kv, D, layout, out_dtype,
                                      causal, scale, descale_q, descale_k, descale_v, stream)


def attn_extend_fwd(q, k_pool, v_pool, page_table, kv_lens, o, lse, B, S_q, H_q, H_kv, D,
                    page_size, max_pages_per_seq, num_pages, dtype, causal, scale,
                    stream) -> int:
    """C ``attn_extend_fwd``; pointers and stream as ints.  Returns the status."""
    return lib().attn_extend_fwd(q, k_pool, v_pool, page_table, kv_lens, o, lse, B, S_q, H_q,
                                 H_kv, D, page_size, max_pages_per_seq, num_pages, dtype, causal,
                                 scale, stream)


def attn_decode_fwd(q, k_pool, v_pool, page_table, kv_lens, o, B, H_q, H_kv, D, page_size,
                    max_pages_per_seq, num_pages, num_splits, scale, dtype, stream) -> int:
    """C ``attn_decode_fwd``; pointers and stream as ints.  Returns the status."""
    return lib().attn_decode_fwd(q, k_pool, v_pool, page_table, kv_lens, o, B, H_q, H_kv, D,
                                 page_size, max_pages_per_seq, num_pages, num_splits, scale,
                                 dtype, stream)


def attn_decode_fwd_noalloc(q, k_pool, v_pool, page_table, kv_lens, o, B, H_q, H_kv, D,
                            page_size, max_pages_per_seq, num_pages, num_splits, scale, dtype,
                            stream) -> int:
    """C ``attn_decode_fwd_noalloc``: decode with its split partials in the
    library's fixed 16 MiB device array, for callers that cannot allocate
    (graph capture, framework-owned memory pools, allocation-free serving
    loops).  Pointers and stream as ints.  Returns the status."""
    return lib().attn_decode_fwd_noalloc(q, k_pool, v_pool, page_table, kv_lens, o, B, H_q,
                                         H_kv, D, page_size, max_pages_per_seq, num_pages,
                                         num_splits, scale, dtype, stream)


def attn_last_error() -> str:
    return last_error()


def attn_device_error(clear: bool = True) -> int:
    """Synchronize, then return (and clear) the device error word; 0 means none."""
    w = ctypes.c_int(0)
    lib().attn_device_error(ctypes.byref(w), 1 if clear else 0)
    return w.value


def attn_set_wait_limit_ns(ns: int) -> None:
    lib().attn_set_wait_limit_ns(ns)


def attn_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Launch a wait that nothing completes; after ``limit_ns`` it records a
    timeout (site 900) in the device error word."""
    _check(lib().attn_selftest_wait_timeout(limit_ns, _stream_handle(stream)))


def attn_release_workspace() -> int:
    return lib().attn_release_workspace()


def attn_version() -> str:
    return lib().attn_version().decode()


# ---------------------------------------------------------- torch wrappers


def _torch():
    import torch  # noqa: PLC0415 - torch is only the memory/stream provider

    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return ATTN_F16
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    raise TypeError("attention tensors must be float16 or bfloat16, got %s" % t.dtype)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _stream_handle(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def prefill(q, k, v, *, causal: bool = False, scale: float | None = None,
            layout: str = "bhsd", out=None, lse=None, return_lse: bool = False, stream=None):
    """Attention forward over torch CUDA tensors.

    ``layout="bhsd"``: q [B,H,S_q,D], k/v [B,H,S_kv,D]; ``"bshd"``: q [B,S_q,H,D],
    k/v [B,S_kv,H,D].  Returns ``o`` (and ``lse`` [B,H,S_q] fp32 if requested).
    """
    torch = _torch()
    _require_cuda(q, k, v, out, lse)
    if layout == "bhsd":
        B, H, S_q, D = q.shape
        S_kv = k.shape[2]
        code = ATTN_BHSD
    elif layout == "bshd":
        B, S_q, H, D = q.shape
        S_kv = k.shape[1]
        code = ATTN_BSHD
    else:
        raise ValueError("layout must be 'bhsd' or 'bshd'")
    if k.shape != v.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k and v must match each other and q's dtype")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, H, S_q), device=q.device, dtype=torch.float32)
    _check(attn_prefill_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            lse.data_ptr() if lse is not None else None, B, H, S_q, S_kv, D,
                            code, _dtype_code(q), int(bool(causal)), float(scale),
                            _stream_handle(stream)))
    return (out, lse) if return_lse else out


def mqa_logits_fp8(q, kv, kv_scale, weights, window_start, window_end, *,
                   clean_logits: bool = True, out=None, stream=None):
    """FP8 MQA logits over torch CUDA tensors: ``q`` [S_q,H,D] and ``kv``
    [S_kv,D] E4M3 (float8_e4m3fn or uint8 codes), ``kv_scale`` [S_kv] and
    ``weights`` [S_q,H] fp32, windows [S_q] int32.  Returns fp32 logits
    [S_q,S_kv] (``out`` may be a preallocated [S_q, >= S_kv] fp32 tensor)."""
    torch = _torch()
    _require_cuda(q, kv, kv_scale, weights, window_start, window_end)
    S_q, H, D = q.shape
    S_kv = kv.shape[0]
    if out is None:
        out = torch.empty((S_q, S_kv), device=q.device, dtype=torch.float32)
    if (not out.is_cuda or out.dtype != torch.float32 or out.dim() != 2 or out.stride(1) != 1
            or tuple(out.shape) != (S_q, S_kv)):
        raise ValueError("out must be a CUDA float32 [S_q, S_kv] tensor with unit column stride")
    _check(attn_mqa_logits_fp8(q.data_ptr(), kv.data_ptr(), kv_scale.data_ptr(),
                               weights.data_ptr(), window_start.data_ptr(),
                               window_end.data_ptr(), out.data_ptr(), S_q, S_kv, H, D,
                               out.stride(0), int(bool(clean_logits)), _stream_handle(stream)))
    return out


def prefill_bwd(q, k, v, o, dout, lse, *, causal: bool = False, scale: float | None = None,
                layout: str = "bhsd", dq=None, dk=None, dv=None, delta=None, stream=None):
    """Gradients (dq, dk, dv) of ``o = prefill(q, k, v)`` for the upstream
    gradient ``dout``, given the forward's ``o`` and ``lse``; torch CUDA tensors
    in the forward's layout.  D must be 128.  ``dq``/``dk``/``dv`` and the fp32
    [B,H,S_q] scratch ``delta`` may be passed in preallocated."""
    torch = _torch()
    _require_cuda(q, k, v, o, dout, lse)
    if layout == "bhsd":
        B, H, S_q, D = q.shape
        S_kv = k.shape[2]
        code = ATTN_BHSD
    elif layout == "bshd":
        B, S_q, H, D = q.shape
        S_kv = k.shape[1]
        code = ATTN_BSHD
    else:
        raise ValueError("layout must be 'bhsd' or 'bshd'")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if delta is None:
        delta = torch.empty((B, H, S_q), device=q.device, dtype=torch.float32)
    _require_cuda(dq, dk, dv, delta)
    _check(attn_prefill_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                            dv.data_ptr(), delta.data_ptr(), B, H, S_q, S_kv, D, code,
                            _dtype_code(q), int(bool(causal)), float(scale),
                            _stream_handle(stream)))
    return dq, dk, dv


def prefill_fp8(q, k, v, *, descale_q: float, descale_k: float, descale_v: float,
                causal: bool = False, scale: float | None = None, layout: str = "bhsd",
                out_dtype=None, out=None, lse=None, return_lse: bool = False, stream=None):
    """FP8 (E4M3) attention forward over torch CUDA tensors.

    ``q``, ``k``, ``v``: torch.float8_e4m3fn (or uint8 holding E4M3 codes) in
    the layout's shape; real values are ``descale_x * value``.  ``o`` is
    bfloat16 unless ``out_dtype`` (torch.float16 / torch.bfloat16) says
    otherwise.  D must be 128.
    """
    torch = _torch()
    _require_cuda(q, k, v, out, lse)
    for t in (q, k, v):
        if t.dtype not in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
            raise TypeError("FP8 prefill inputs must be float8_e4m3fn or uint8 codes")
    if layout == "bhsd":
        B, H, S_q, D = q.shape
        S_kv = k.shape[2]
        code = ATTN_BHSD
    elif layout == "bshd":
        B, S_q, H, D = q.shape
        S_kv = k.shape[1]
        code = ATTN_BSHD
    else:
        raise ValueError("layout must be 'bhsd' or 'bshd'")
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty(q.shape, device=q.device,
                          dtype=out_dtype if out_dtype is not None else torch.bfloat16)
    if return_lse and lse is None:
        lse = torch.empty((B, H, S_q), device=q.device, dtype=torch.float32)
    _check(attn_prefill_fp8_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                lse.data_ptr() if lse is not None else None, B, H, S_q, S_kv, D,
                                code, _dtype_code(out), int(bool(causal)), float(scale),
                                float(descale_q), float(descale_k), float(descale_v),
                                _stream_handle(stream)))
    return (out, lse) if return_lse else out


def extend(q, k_pool, v_pool, page_table, kv_lens, *, causal: bool = True,
           scale: float | None = None, num_pages: int | None = None, out=None, lse=None,
           return_lse: bool = False, stream=None):
    """Extend (prefix-cached prefill) over torch CUDA tensors.

    ``q`` [B,S_q,H_q,D]; ``k_pool``/``v_pool`` [num_pages, page_size, H_kv, D];
    ``page_table`` [B, max_pages] int32; ``kv_lens`` [B] int32 = cached prefix
    plus the S_q new tokens (already written to the pool).  Returns ``o``
    [B,S_q,H_q,D] (and ``lse`` [B,H_q,S_q] fp32 if requested).
    """
    torch = _torch()
    _require_cuda(q, k_pool, v_pool, kv_lens, page_table, out, lse)
    B, S_q, H_q, D = q.shape
    n_pages, page_size, H_kv, D2 = k_pool.shape
    if D2 != D or v_pool.shape != k_pool.shape:
        raise ValueError("k_pool/v_pool must be [pages, page_size, H_kv, D]")
    if k_pool.dtype != q.dtype or v_pool.dtype != q.dtype:
        raise ValueError("k_pool and v_pool must have q's dtype")
    if kv_lens.dtype != torch.int32 or page_table.dtype != torch.int32:
        raise TypeError("kv_lens and page_table must be int32")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, H_q, S_q), device=q.device, dtype=torch.float32)
    _check(attn_extend_fwd(q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
                           page_table.data_ptr(), kv_lens.data_ptr(), out.data_ptr(),
                           lse.data_ptr() if lse is not None else None, B, S_q, H_q, H_kv, D,
                           page_size, page_table.shape[1],
                           n_pages if num_pages is None else num_pages, _dtype_code(q),
                           int(bool(causal)), float(scale), _stream_handle(stream)))
    return (out, lse) if return_lse else out


def decode(q, k_pool, v_pool, kv_lens, *, page_table=None, num_pages: int | None = None,
           num_splits: int = 0, scale: float | None = None, out=None, stream=None):
    """Decode attention over torch CUDA tensors.

    ``q`` [B,H_q,D]; paged: ``k_pool``/``v_pool`` [num_pages, page_size, H_kv, D] and
    ``page_table`` [B, max_pages] int32; contiguous (``page_table=None``):
    ``k_pool``/``v_pool`` [B, S_max, H_kv, D].  ``kv_lens`` [B] int32 (CUDA).
    """
    torch = _torch()
    _require_cuda(q, k_pool, v_pool, kv_lens, page_table, out)
    B, H_q, D = q.shape
    n_pages, page_size, H_kv, D2 = k_pool.shape
    if D2 != D or v_pool.shape != k_pool.shape:
        raise ValueError("k_pool/v_pool must be [pages, page_size, H_kv, D]")
    if kv_lens.dtype != torch.int32 or (page_table is not None and page_table.dtype != torch.int32):
        raise TypeError("kv_lens and page_table must be int32")
    if page_table is not None:
        max_pages = page_table.shape[1]
        num_pages = n_pages if num_pages is None else num_pages
    else:
        max_pages = 1
        num_pages = B
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    _check(attn_decode_fwd(q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
                           page_table.data_ptr() if page_table is not None else None,
                           kv_lens.data_ptr(), out.data_ptr(), B, H_q, H_kv, D, page_size,
                           max_pages, num_pages, int(num_splits), float(scale), _dtype_code(q),
                           _stream_handle(stream)))
    return out


def check_device_error() -> None:
    """Raise AttnError if any kernel recorded a device error (synchronizes)."""
    w = ctypes.c_int(0)
    st = lib().attn_device_error(ctypes.byref(w), 1)
    if st != ATTN_OK:
        raise AttnError(st, last_error())


__all__ = [n for n in dir() if n.startswith(("attn_", "ATTN_"))] + [
    "AttnError", "prefill", "prefill_bwd", "mqa_logits_fp8", "prefill_fp8", "extend", "decode", "lib", "library_path", "check_device_error", "EXPORTED"]
