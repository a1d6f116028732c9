"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws random tensors and
lays out KV pages.  Both the CUDA path's tests and the float64 oracle are fed
from it, so they see bit-identical inputs.

Recipe (every draw uses a CPU ``torch.Generator`` seeded with ``seed``):

* prefill: Q, K, V drawn in that order as float32 ``randn`` in the layout's
  own shape ([B,H,S,D] for BHSD, [B,S,H,D] for BSHD), multiplied by ``std``
  (exact for 0.5) and rounded to nearest-even into fp16/bf16.
* decode: first ``kv_lens`` (``randint`` uniform on [kv_min, kv_max]), then
  Q [B,H_q,D], then for each sequence b in order its K rows then its V rows
  ([kv_len_b, H_kv, D], float32 ``randn`` rounded to bf16/fp16), then the page
  permutation (``randperm`` over the data pages).
  Contiguous KV is [B, S_max, H_kv, D]; rows at or past ``kv_len_b`` hold the
  finite poison value 1e4.  Paged KV is a pool of 16-token pages
  [num_pages, page_size, H_kv, D]: sequence b owns ceil(kv_len_b/page_size)
  data pages placed by the permutation, one extra poison page (all 1e4) is
  appended, unused page-table entries point at it, and page tail slots hold
  1e4 too, so a masking bug is loud but never reads outside the pool.
* backward: Q, K, V drawn as for prefill, then the upstream gradient dO
  (q's shape, float32 ``randn`` times ``std``, rounded to the dtype).
* FP8 prefill: Q, K, V drawn as for prefill in float32 (times ``std``), then
  each tensor is quantized on its own: descale = max|x| / 448 and the E4M3
  codes are ``(x / descale)`` rounded by PyTorch's float8_e4m3fn conversion
  (round to nearest even).  The codes and the three descale factors are the
  inputs; nothing of the attention arithmetic happens here.
* FP8 MQA logits: q ``randn`` [S_q,H,D] rounded to E4M3 (no separate scale),
  then kv ``randn`` [S_kv,D] quantized per row (kv_scale[j] = max|row|/448,
  codes = row / kv_scale), then weights ``randn`` [S_q,H] / sqrt(H) in
  float32, then the windows of the chosen kind (below, in ``mqa_windows``).
* extend (prefill of new tokens against a paged cache): first the cached
  prefix lengths (``randint`` uniform on [prefix_min, prefix_max]) unless
  given, ``kv_len_b = prefix_b + S_q``; then Q [B,S_q,H_q,D]; then per
  sequence its K rows then V rows; then the page permutation, poison page and
  poison tails exactly as for paged decode.

The five named workloads follow the configurations this library is measured
on; their shapes mirror the pages' LLM attention workloads (e.g. the
Llama-2-13B-like 40-head, D=128 shape of the WAVE MLSys 2026 summary,
Attention (prefill) and Figure 8).  No public suite or dataset is involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

POISON = 1.0e4

_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class PrefillCase:
    name: str
    B: int
    H: int
    S_q: int
    S_kv: int
    D: int
    layout: str  # "bhsd" or "bshd"
    dtype: str  # "fp16" or "bf16"
    causal: bool
    std: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def flops(self) -> float:
        """Algorithmic FLOPs: 4*D per visible (query, key) pair (QK^T and PV)."""
        return 4.0 * self.B * self.H * self.D * visible_pairs(self.S_q, self.S_kv, self.causal)

    def bytes(self) -> int:
        el = 2
        return el * self.B * self.H * self.D * (2 * self.S_q + 2 * self.S_kv)


@dataclass(frozen=True)
class DecodeCase:
    name: str
    B: int
    H_q: int
    H_kv: int
    D: int
    kv_min: int
    kv_max: int
    S_max: int
    paged: bool
    page_size: int = 16
    dtype: str = "bf16"
    seed: int = 0
    num_splits: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def max_pages(self) -> int:
        return -(-self.S_max // self.page_size)


@dataclass(frozen=True)
class ExtendCase:
    """S_q new query tokens per sequence against ``prefix + S_q`` cached keys
    in a paged pool (bottom-right causal per sequence when ``causal``)."""
    name: str
    B: int
    S_q: int
    H_q: int
    H_kv: int
    D: int
    prefix_min: int
    prefix_max: int
    page_size: int = 16
    dtype: str = "bf16"
    causal: bool = True
    std: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def max_pages(self) -> int:
        return -(-(self.prefix_max + self.S_q) // self.page_size)


def visible_pairs(S_q: int, S_kv: int, causal: bool) -> int:
    """Number of (query, key) pairs the mask leaves visible (bottom-right causal)."""
    if not causal:
        return S_q * S_kv
    off = S_kv - S_q
    total = 0
    # row i sees keys 0 .. min(S_kv-1, i+off)
    for i in range(S_q):
        total += max(0, min(S_kv, i + off + 1))
    return total


# The five workloads (tiny oracle case, two prefill shapes, two decode shapes).
C1 = PrefillCase("prefill_tiny_bhsd_fp16", 1, 2, 128, 128, 64, "bhsd", "fp16", False)
C2 = PrefillCase("prefill_bhsd_fp16_b4_h32_s4096_d128", 4, 32, 4096, 4096, 128, "bhsd", "fp16", False)
C2_CAUSAL = PrefillCase("prefill_bhsd_fp16_b4_h32_s4096_d128_causal", 4, 32, 4096, 4096, 128,
                        "bhsd", "fp16", True)
C3 = PrefillCase("prefill_bshd_bf16_b8_h40_s2048_d128_causal", 8, 40, 2048, 2048, 128, "bshd",
                 "bf16", True, std=0.5)
C4 = DecodeCase("decode_contig_bf16_b32_hq32_hkv8_d128", 32, 32, 8, 128, 1024, 32768, 32768,
                paged=False)
C5 = DecodeCase("decode_paged16_bf16_b32_hq32_hkv8_d128", 32, 32, 8, 128, 1, 32768, 32768,
                paged=True)


@dataclass(frozen=True)
class Fp8PrefillCase:
    """Prefill on E4M3 inputs with per-tensor descale factors; O in ``out_dtype``."""
    name: str
    B: int
    H: int
    S_q: int
    S_kv: int
    D: int
    layout: str
    causal: bool
    out_dtype: str = "bf16"
    std: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def flops(self) -> float:
        return 4.0 * self.B * self.H * self.D * visible_pairs(self.S_q, self.S_kv, self.causal)


# Backward of the C2 forward shape (bf16, non-causal and causal).
C8 = PrefillCase("prefill_bwd_bhsd_bf16_b4_h32_s4096_d128", 4, 32, 4096, 4096, 128, "bhsd", "bf16",
                 False)
C8_CAUSAL = PrefillCase("prefill_bwd_bhsd_bf16_b4_h32_s4096_d128_causal", 4, 32, 4096, 4096, 128,
                        "bhsd", "bf16", True)

# The BHSD prefill shape of C2 with E4M3 inputs (the pages' "FAv3 - FP8" item).
C7 = Fp8PrefillCase("prefill_fp8e4m3_bhsd_b4_h32_s4096_d128", 4, 32, 4096, 4096, 128, "bhsd",
                    False)
C7_CAUSAL = Fp8PrefillCase("prefill_fp8e4m3_bhsd_b4_h32_s4096_d128_causal", 4, 32, 4096, 4096,
                           128, "bhsd", True)

@dataclass(frozen=True)
class MqaCase:
    """FP8 MQA logits: S_q query rows of H heads against S_kv shared keys."""
    name: str
    S_q: int
    S_kv: int
    H: int
    D: int
    window: str  # causal | cp | misaligned | empty | past_end
    clean_logits: bool = True
    seed: int = 0

    def flops(self, start, end) -> float:
        """2*H*D per in-window (row, key) pair (the per-head dot products)."""
        lo = start.clamp(min=0)
        hi = end.clamp(max=self.S_kv)
        return 2.0 * self.H * self.D * float((hi - lo).clamp(min=0).sum())


# Long-context indexer shape of the page's sweep (2048 x 131072 is its largest;
# this one keeps the fp32 output at 256 MiB): 1024 rows x 65536 keys, 64 heads, D=128.
C9 = MqaCase("mqa_logits_fp8_sq1024_skv65536_h64_d128_causal", 1024, 65536, 64, 128, "causal")

# Prefix-cached prefill: 8 requests of 1024 new tokens each on top of cached
# prefixes of up to 15360 tokens, Llama-3-8B-like GQA heads, 16-token pages.
C6 = ExtendCase("extend_paged16_bf16_b8_sq1024_hq32_hkv8_d128_causal", 8, 1024, 32, 8, 128, 0,
                15360)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _randn(g, shape, std, dtype):
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def prefill_shape(B, H, S, D, layout):
    return (B, H, S, D) if layout == "bhsd" else (B, S, H, D)


def make_prefill_bwd(case: PrefillCase):
    """Return CPU tensors (q, k, v, dout) for a backward case (q, k, v exactly as
    make_prefill draws them)."""
    g = _gen(case.seed)
    dt = _DTYPES[case.dtype]
    q = _randn(g, prefill_shape(case.B, case.H, case.S_q, case.D, case.layout), case.std, dt)
    k = _randn(g, prefill_shape(case.B, case.H, case.S_kv, case.D, case.layout), case.std, dt)
    v = _randn(g, prefill_shape(case.B, case.H, case.S_kv, case.D, case.layout), case.std, dt)
    do = _randn(g, prefill_shape(case.B, case.H, case.S_q, case.D, case.layout), case.std, dt)
    return q, k, v, do


def make_prefill(case: PrefillCase):
    """Return CPU tensors (q, k, v) for a prefill case."""
    g = _gen(case.seed)
    dt = _DTYPES[case.dtype]
    q = _randn(g, prefill_shape(case.B, case.H, case.S_q, case.D, case.layout), case.std, dt)
    k = _randn(g, prefill_shape(case.B, case.H, case.S_kv, case.D, case.layout), case.std, dt)
    v = _randn(g, prefill_shape(case.B, case.H, case.S_kv, case.D, case.layout), case.std, dt)
    return q, k, v


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor E4M3 quantization: returns (codes as float8_e4m3fn, descale)."""
    amax = float(x.abs().max())
    descale = amax / 448.0 if amax > 0 else 1.0
    return (x / descale).to(torch.float8_e4m3fn), descale


def make_prefill_fp8(case: Fp8PrefillCase):
    """Return (q8, k8, v8, dq, dk, dv): float8_e4m3fn CPU tensors and descales."""
    g = _gen(case.seed)
    qs = prefill_shape(case.B, case.H, case.S_q, case.D, case.layout)
    ks = prefill_shape(case.B, case.H, case.S_kv, case.D, case.layout)
    q = _randn(g, qs, case.std, torch.float32)
    k = _randn(g, ks, case.std, torch.float32)
    v = _randn(g, ks, case.std, torch.float32)
    (q8, dq), (k8, dk), (v8, dv) = quantize_e4m3(q), quantize_e4m3(k), quantize_e4m3(v)
    return q8, k8, v8, dq, dk, dv


@dataclass
class DecodeInputs:
    q: torch.Tensor  # [B, H_q, D]
    k: torch.Tensor  # contiguous [B, S_max, H_kv, D] or pool [P, page_size, H_kv, D]
    v: torch.Tensor
    kv_lens: torch.Tensor  # [B] int32
    page_table: torch.Tensor | None = None  # [B, max_pages] int32
    page_size: int = 0
    max_pages: int = 1
    extra: dict = field(default_factory=dict)

    def kv_bytes(self) -> int:
        """Algorithmic K/V bytes one decode pass must read (kv_len rows per (b, kv head))."""
        H_kv, D = self.k.shape[2], self.k.shape[3]
        el = self.k.element_size()
        return int(self.kv_lens.to(torch.int64).sum().item()) * H_kv * D * el * 2


def make_decode(case: DecodeCase, kv_lens=None) -> DecodeInputs:
    """Return CPU tensors for a decode case (see the module docstring recipe)."""
    g = _gen(case.seed)
    dt = _DTYPES[case.dtype]
    if kv_lens is None:
        kv_lens = torch.randint(case.kv_min, case.kv_max + 1, (case.B,), generator=g,
                                dtype=torch.int64)
    kv_lens = torch.as_tensor(kv_lens, dtype=torch.int64)
    assert int(kv_lens.max()) <= case.S_max and int(kv_lens.min()) >= 0
    q = _randn(g, (case.B, case.H_q, case.D), 1.0, dt)
    rows_k, rows_v = [], []
    for b in range(case.B):
        n = int(kv_lens[b])
        rows_k.append(_randn(g, (n, case.H_kv, case.D), 1.0, dt))
        rows_v.append(_randn(g, (n, case.H_kv, case.D), 1.0, dt))
    lens32 = kv_lens.to(torch.int32)
    if not case.paged:
        k = torch.full((case.B, case.S_max, case.H_kv, case.D), POISON, dtype=dt)
        v = torch.full((case.B, case.S_max, case.H_kv, case.D), POISON, dtype=dt)
        for b in range(case.B):
            n = int(kv_lens[b])
            k[b, :n] = rows_k[b]
            v[b, :n] = rows_v[b]
        return DecodeInputs(q, k, v, lens32, None, case.S_max, 1)
    ps = case.page_size
    k, v, page_table = _place_pages(g, rows_k, rows_v, kv_lens, ps, case.max_pages, case.H_kv,
                                    case.D, dt)
    return DecodeInputs(q, k, v, lens32, page_table, ps, case.max_pages)


def contiguous_view_of(inp: DecodeInputs, S_max: int | None = None) -> DecodeInputs:
    """Re-lay a paged DecodeInputs as contiguous [B, S_max, H_kv, D] (poison past kv_len).

    Pure data movement: used by tests that check paged == contiguous."""
    if inp.page_table is None:
        return inp
    B = inp.q.shape[0]
    ps = inp.page_size
    S_max = S_max or inp.max_pages * ps
    H_kv, D = inp.k.shape[2], inp.k.shape[3]
    k = torch.full((B, S_max, H_kv, D), POISON, dtype=inp.k.dtype)
    v = torch.full((B, S_max, H_kv, D), POISON, dtype=inp.v.dtype)
    for b in range(B):
        n = int(inp.kv_lens[b])
        for p in range(-(-n // ps)):
            lo, hi = p * ps, min(n, (p + 1) * ps)
            phys = int(inp.page_table[b, p])
            k[b, lo:hi] = inp.k[phys, : hi - lo]
            v[b, lo:hi] = inp.v[phys, : hi - lo]
    return DecodeInputs(inp.q, k, v, inp.kv_lens, None, S_max, 1)


@dataclass
class ExtendInputs:
    q: torch.Tensor  # [B, S_q, H_q, D]
    k: torch.Tensor  # pool [num_pages, page_size, H_kv, D]
    v: torch.Tensor
    kv_lens: torch.Tensor  # [B] int32, prefix + S_q
    page_table: torch.Tensor  # [B, max_pages] int32
    page_size: int
    max_pages: int

    def visible_pairs(self, causal: bool) -> int:
        S_q = self.q.shape[1]
        return sum(visible_pairs(S_q, int(n), causal) for n in self.kv_lens.tolist())

    def flops(self, causal: bool) -> float:
        """Algorithmic FLOPs: 4*D per visible (query, key) pair and query head."""
        H_q, D = self.q.shape[2], self.q.shape[3]
        return 4.0 * H_q * D * self.visible_pairs(causal)


def _place_pages(g, rows_k, rows_v, kv_lens, ps, max_pages, H_kv, D, dt):
    """Scatter per-sequence rows into a permuted page pool (shared by paged
    decode and extend): returns (k_pool, v_pool, page_table)."""
    B = len(rows_k)
    pages_per_seq = [-(-int(n) // ps) for n in kv_lens.tolist()]
    n_data = sum(pages_per_seq)
    perm = torch.randperm(n_data, generator=g)
    poison_page = n_data
    k = torch.full((n_data + 1, ps, H_kv, D), POISON, dtype=dt)
    v = torch.full((n_data + 1, ps, H_kv, D), POISON, dtype=dt)
    page_table = torch.full((B, max_pages), poison_page, dtype=torch.int32)
    cursor = 0
    for b in range(B):
        n = int(kv_lens[b])
        for p in range(pages_per_seq[b]):
            phys = int(perm[cursor])
            cursor += 1
            page_table[b, p] = phys
            lo, hi = p * ps, min(n, (p + 1) * ps)
            k[phys, : hi - lo] = rows_k[b][lo:hi]
            v[phys, : hi - lo] = rows_v[b][lo:hi]
    return k, v, page_table


def make_extend(case: ExtendCase, prefix_lens=None) -> ExtendInputs:
    """Return CPU tensors for an extend case (see the module docstring recipe)."""
    g = _gen(case.seed)
    dt = _DTYPES[case.dtype]
    if prefix_lens is None:
        prefix_lens = torch.randint(case.prefix_min, case.prefix_max + 1, (case.B,), generator=g,
                                    dtype=torch.int64)
    prefix_lens = torch.as_tensor(prefix_lens, dtype=torch.int64)
    assert int(prefix_lens.min()) >= 0 and int(prefix_lens.max()) <= case.prefix_max
    kv_lens = prefix_lens + case.S_q
    q = _randn(g, (case.B, case.S_q, case.H_q, case.D), case.std, dt)
    rows_k, rows_v = [], []
    for b in range(case.B):
        n = int(kv_lens[b])
        rows_k.append(_randn(g, (n, case.H_kv, case.D), case.std, dt))
        rows_v.append(_randn(g, (n, case.H_kv, case.D), case.std, dt))
    k, v, pt = _place_pages(g, rows_k, rows_v, kv_lens, case.page_size, case.max_pages,
                            case.H_kv, case.D, dt)
    return ExtendInputs(q, k, v, kv_lens.to(torch.int32), pt, case.page_size, case.max_pages)


def mqa_windows(kind: str, S_q: int, S_kv: int, g: torch.Generator):
    """[start, end) per query row for the window kinds of the MQA-logits
    sweep; `g` draws the random ones.
      causal:     [0, i + S_kv - S_q + 1)            (bottom-right)
      cp:         the second half of the causal window (a context-parallel
                  shard that sees a suffix of its prefix)
      misaligned: random start <= end inside [0, S_kv], not tile-aligned
      empty:      end == start (random start)
      past_end:   start >= S_kv
    """
    i = torch.arange(S_q, dtype=torch.int64)
    causal_end = (i + S_kv - S_q + 1).clamp(min=0, max=S_kv)
    if kind == "causal":
        start, end = torch.zeros_like(i), causal_end
    elif kind == "cp":
        start, end = causal_end // 2, causal_end
    elif kind == "misaligned":
        a = torch.randint(0, S_kv + 1, (S_q,), generator=g)
        b = torch.randint(0, S_kv + 1, (S_q,), generator=g)
        start, end = torch.minimum(a, b), torch.maximum(a, b)
    elif kind == "empty":
        start = torch.randint(0, S_kv + 1, (S_q,), generator=g)
        end = start.clone()
    elif kind == "past_end":
        start = S_kv + torch.randint(0, 64, (S_q,), generator=g)
        end = start + torch.randint(0, 64, (S_q,), generator=g)
    else:
        raise ValueError(kind)
    return start.to(torch.int32), end.to(torch.int32)


def make_mqa(case: MqaCase):
    """Return (q8 [S_q,H,D] e4m3, kv8 [S_kv,D] e4m3, kv_scale [S_kv] f32,
    weights [S_q,H] f32, start, end [S_q] int32) on the CPU."""
    g = _gen(case.seed)
    q8 = torch.randn((case.S_q, case.H, case.D), generator=g).to(torch.float8_e4m3fn)
    kv = torch.randn((case.S_kv, case.D), generator=g)
    amax = kv.abs().amax(dim=1).clamp(min=1e-6)
    kv_scale = (amax / 448.0).to(torch.float32)
    kv8 = (kv / kv_scale[:, None]).to(torch.float8_e4m3fn)
    w = torch.randn((case.S_q, case.H), generator=g) / math.sqrt(case.H)
    start, end = mqa_windows(case.window, case.S_q, case.S_kv, g)
    return q8, kv8, kv_scale, w.to(torch.float32), start, end
