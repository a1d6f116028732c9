"""Float64 CPU oracle for the attention forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg (``bench.py``) may import this package.  The product path
(``attention_flash_attn_fwd_gb300``) never imports, loads or calls it, and it
imports nothing from the product.

The arithmetic lives in ``attn_oracle.c`` (plain C, float64, POSIX threads);
this module compiles it with gcc, widens inputs exactly to float64 and calls
it through ctypes.  What the oracle computes and which passages it follows
are stated at the top of ``attn_oracle.c``:

* prefill: ``O = softmax(scale * Q K^T + causal mask) V`` over BHSD or BSHD
  tensors, bottom-right causal alignment, ``lse = ln sum exp`` per row
  (Wave February 2025 Release, "Prefill attention kernel"; WAVE MLSys 2026
  summary, Attention (prefill), Figures 2-4, and Assumption 1 on BHSD/BSHD);
* decode: one query per head against a sequence's first ``kv_len`` keys read
  through a page table, grouped-query heads ``g = h // (H_q // H_kv)``
  (Wave February 2025 Release, FlashDecoding list: paged flash decoding and
  the fake-page-table test fixture);
* extend: S_q new queries per sequence against its ``kv_len`` keys in the
  paged pool, bottom-right causal per sequence (Wave February 2025 Release,
  "Extend Attention"; WAVE MLSys 2026 summary, Integration: SGLang extend);
* FP8 prefill: the prefill definition on E4M3 codes times per-tensor descale
  factors (Wave February 2025 Release, EvoFormer list, "FAv3 - FP8"), E4M3 decoded from the
  OCP 8-bit floating point definition;
* backward: dQ, dK, dV of the prefill definition by the chain rule
  (Wave February 2025 Release, EvoFormer list, "Backward Flash Attention");
* FP8 MQA logits: sum over heads of w * ReLU(kv_scale * q.k) inside each
  row's key window (aiter PR 7412, "FP8 MQA logits"; the formula is a
  reading, stated in ``attn_oracle.c``).

Every function here is pinned by ``tests/test_oracle.py`` against library
routines, closed forms and analytic fixtures; no part is left unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

BHSD = 0
BSHD = 1

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``oracle/_build/liboracle.so``.

    Plain ``-O2``: no fast-math, no ``-march=native``, so the same source
    gives the same float64 results on x86_64 and aarch64 hosts.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            L = ctypes.c_long
            lib.oracle_prefill_f64.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, L,
                                               ctypes.c_int, ctypes.c_int,
                                               ctypes.c_double, ctypes.c_int]
            lib.oracle_prefill_f64.restype = ctypes.c_int
            lib.oracle_decode_f64.argtypes = [dp, dp, dp, ip, ip, dp, dp, L, L, L,
                                              L, L, L, ctypes.c_double, ctypes.c_int]
            lib.oracle_decode_f64.restype = ctypes.c_int
            lib.oracle_extend_f64.argtypes = [dp, dp, dp, ip, ip, dp, dp, L, L, L, L, L, L,
                                              L, ctypes.c_int, ctypes.c_double, ctypes.c_int]
            lib.oracle_extend_f64.restype = ctypes.c_int
            lib.oracle_e4m3_decode.argtypes = [ctypes.POINTER(ctypes.c_uint8), dp, L]
            lib.oracle_e4m3_decode.restype = None
            lib.oracle_prefill_bwd_f64.argtypes = [dp, dp, dp, dp, dp, dp, dp, L, L, L, L, L,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                   ctypes.c_int]
            lib.oracle_prefill_bwd_f64.restype = ctypes.c_int
            lib.oracle_mqa_logits_f64.argtypes = [dp, dp, dp, dp, ip, ip, dp, L, L, L, L, L,
                                                  ctypes.c_int, ctypes.c_int]
            lib.oracle_mqa_logits_f64.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    """Threads the oracle uses by default: every core this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


def _f64(x) -> np.ndarray:
    """Exact widening of a numpy array or torch tensor (any float dtype) to a
    contiguous float64 numpy array."""
    if hasattr(x, "detach"):  # torch tensor, possibly fp16/bf16
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def prefill(q, k, v, *, causal: bool, scale: float, layout: int = BHSD,
            n_threads: int | None = None):
    """Attention forward in float64.

    ``q``: [B,H,S_q,D] (BHSD) or [B,S_q,H,D] (BSHD); ``k``, ``v``: the same
    layout with S_kv rows.  Returns ``(o, lse)`` as float64 numpy arrays:
    ``o`` in q's layout, ``lse`` [B,H,S_q] natural-log (``-inf`` for a row
    with no visible key, whose ``o`` is 0).
    """
    q64, k64, v64 = _f64(q), _f64(k), _f64(v)
    if layout == BHSD:
        B, H, S_q, D = q64.shape
        S_kv = k64.shape[2]
        kv_shape = (B, H, S_kv, D)
    elif layout == BSHD:
        B, S_q, H, D = q64.shape
        S_kv = k64.shape[1]
        kv_shape = (B, S_kv, H, D)
    else:
        raise ValueError("layout must be BHSD (0) or BSHD (1)")
    if k64.shape != kv_shape or v64.shape != kv_shape:
        raise ValueError("k and v must be %r, got %r and %r" % (kv_shape, k64.shape, v64.shape))
    o = np.zeros(q64.shape, dtype=np.float64)
    lse = np.zeros((B, H, S_q), dtype=np.float64)
    rc = _load().oracle_prefill_f64(_dptr(q64), _dptr(k64), _dptr(v64), _dptr(o), _dptr(lse),
                                    B, H, S_q, S_kv, D, int(layout), int(bool(causal)),
                                    float(scale), int(n_threads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_prefill_f64 failed (rc=%d)" % rc)
    return o, lse


def decode(q, k_pool, v_pool, kv_lens, *, scale: float, page_table=None,
           n_threads: int | None = None):
    """Seq_len=1 attention over a paged (or contiguous) KV cache, float64.

    ``q``: [B,H_q,D].  Paged: ``k_pool``/``v_pool`` [num_pages, page_size,
    H_kv, D] and ``page_table`` [B, max_pages] int32.  Contiguous
    (``page_table is None``): ``k_pool``/``v_pool`` [B, S_max, H_kv, D].
    ``kv_lens``: [B] int32.  Returns ``(o [B,H_q,D], lse [B,H_q])``.
    """
    q64, k64, v64 = _f64(q), _f64(k_pool), _f64(v_pool)
    lens = _i32(kv_lens)
    B, H_q, D = q64.shape
    _, page_size, H_kv, D2 = k64.shape
    if D2 != D or v64.shape != k64.shape:
        raise ValueError("k_pool/v_pool shape mismatch")
    if lens.shape != (B,):
        raise ValueError("kv_lens must be [B]")
    pt = None
    max_pages = 1
    if page_table is not None:
        pt = _i32(page_table)
        if pt.ndim != 2 or pt.shape[0] != B:
            raise ValueError("page_table must be [B, max_pages]")
        max_pages = pt.shape[1]
    elif k64.shape[0] != B:
        raise ValueError("contiguous k/v must be [B, S_max, H_kv, D]")
    o = np.zeros((B, H_q, D), dtype=np.float64)
    lse = np.zeros((B, H_q), dtype=np.float64)
    rc = _load().oracle_decode_f64(_dptr(q64), _dptr(k64), _dptr(v64), _iptr(pt), _iptr(lens),
                                   _dptr(o), _dptr(lse), B, H_q, H_kv, D, page_size, max_pages,
                                   float(scale), int(n_threads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_decode_f64 failed (rc=%d)" % rc)
    return o, lse


def extend(q, k_pool, v_pool, page_table, kv_lens, *, causal: bool, scale: float,
           n_threads: int | None = None):
    """Prefill of S_q new queries per sequence against a paged KV cache, float64.

    ``q``: [B,S_q,H_q,D]; ``k_pool``/``v_pool``: [num_pages, page_size, H_kv, D];
    ``page_table``: [B, max_pages] int32; ``kv_lens``: [B] int32 (cached keys
    including the new tokens).  Returns ``(o [B,S_q,H_q,D], lse [B,H_q,S_q])``.
    """
    q64, k64, v64 = _f64(q), _f64(k_pool), _f64(v_pool)
    pt, lens = _i32(page_table), _i32(kv_lens)
    B, S_q, H_q, D = q64.shape
    _, page_size, H_kv, D2 = k64.shape
    if D2 != D or v64.shape != k64.shape or pt.ndim != 2 or pt.shape[0] != B:
        raise ValueError("shape mismatch")
    o = np.zeros(q64.shape, dtype=np.float64)
    lse = np.zeros((B, H_q, S_q), dtype=np.float64)
    rc = _load().oracle_extend_f64(_dptr(q64), _dptr(k64), _dptr(v64), _iptr(pt), _iptr(lens),
                                   _dptr(o), _dptr(lse), B, S_q, H_q, H_kv, D, page_size,
                                   pt.shape[1], int(bool(causal)), float(scale),
                                   int(n_threads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_extend_f64 failed (rc=%d)" % rc)
    return o, lse


def decode_e4m3(codes) -> np.ndarray:
    """Float64 values of E4M3 codes (a uint8 numpy array or a torch uint8 /
    float8_e4m3fn tensor), same shape."""
    if hasattr(codes, "detach"):
        t = codes.detach().to("cpu")
        if t.dtype != __import__("torch").uint8:
            t = t.view(__import__("torch").uint8)
        codes = t.numpy()
    u8 = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(u8.shape, dtype=np.float64)
    _load().oracle_e4m3_decode(u8.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), _dptr(out),
                               u8.size)
    return out


def prefill_fp8(q, k, v, *, descale_q: float, descale_k: float, descale_v: float, causal: bool,
                scale: float, layout: int = BHSD, n_threads: int | None = None):
    """FP8 prefill in float64: Q, K, V are E4M3 codes (layouts as ``prefill``),
    real values descale_x * value(code).  Returns ``(o, lse)`` like ``prefill``."""
    return prefill(decode_e4m3(q) * float(descale_q), decode_e4m3(k) * float(descale_k),
                   decode_e4m3(v) * float(descale_v), causal=causal, scale=scale, layout=layout,
                   n_threads=n_threads)


def prefill_bwd(q, k, v, dout, *, causal: bool, scale: float, layout: int = BHSD,
                n_threads: int | None = None):
    """Gradients (dq, dk, dv) in float64 of ``O = prefill(q, k, v)`` for the
    upstream gradient ``dout`` (q's shape); layouts as ``prefill``."""
    q64, k64, v64, do64 = _f64(q), _f64(k), _f64(v), _f64(dout)
    if layout == BHSD:
        B, H, S_q, D = q64.shape
        S_kv = k64.shape[2]
    elif layout == BSHD:
        B, S_q, H, D = q64.shape
        S_kv = k64.shape[1]
    else:
        raise ValueError("layout must be BHSD (0) or BSHD (1)")
    if do64.shape != q64.shape or k64.shape != v64.shape:
        raise ValueError("shape mismatch")
    dq = np.zeros(q64.shape, dtype=np.float64)
    dk = np.zeros(k64.shape, dtype=np.float64)
    dv = np.zeros(v64.shape, dtype=np.float64)
    rc = _load().oracle_prefill_bwd_f64(_dptr(q64), _dptr(k64), _dptr(v64), _dptr(do64),
                                        _dptr(dq), _dptr(dk), _dptr(dv), B, H, S_q, S_kv, D,
                                        int(layout), int(bool(causal)), float(scale),
                                        int(n_threads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_prefill_bwd_f64 failed (rc=%d)" % rc)
    return dq, dk, dv


def mqa_logits(q, kv, kv_scale, weights, start, end, *, clean_logits: bool, out=None,
               n_threads: int | None = None):
    """FP8 MQA logits in float64 (inputs already decoded to numbers):
    ``q`` [S_q,H,D], ``kv`` [S_kv,D], ``kv_scale`` [S_kv], ``weights`` [S_q,H],
    ``start``/``end`` [S_q] int32.  Returns logits [S_q,S_kv]; entries outside
    a row's window are -inf with ``clean_logits``, else those of ``out``
    (NaN if ``out`` is None)."""
    q64, kv64, sc64, w64 = _f64(q), _f64(kv), _f64(kv_scale), _f64(weights)
    st, en = _i32(start), _i32(end)
    S_q, H, D = q64.shape
    S_kv = kv64.shape[0]
    res = np.full((S_q, S_kv), np.nan) if out is None else np.array(_f64(out), copy=True)
    rc = _load().oracle_mqa_logits_f64(_dptr(q64), _dptr(kv64), _dptr(sc64), _dptr(w64),
                                       _iptr(st), _iptr(en), _dptr(res), S_q, S_kv, H, D, S_kv,
                                       int(bool(clean_logits)),
                                       int(n_threads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_mqa_logits_f64 failed (rc=%d)" % rc)
    return res
