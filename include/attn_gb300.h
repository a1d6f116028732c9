/*
 * attn_gb300.h -- C ABI of the GB300 (sm_103a) fused attention forward library.
 *
 * The library computes the scaled-dot-product attention forward
 *
 *     O = softmax(scale * Q K^T + causal mask) V
 *
 * in two forms:
 *   - prefill, over BHSD or BSHD tensors ("Prefill attention kernel" in the
 *     Wave February 2025 Release, FlashDecoding list; WAVE MLSys 2026 summary,
 *     Attention (prefill), Figures 2-4, and its Assumption 1: BSHD only swaps
 *     the boundary indexing of BHSD);
 *   - seq_len = 1 flash decoding with split KV over a paged or contiguous KV
 *     cache ("Flash Decoding Kernel with paged attention" and "... without
 *     paged attention ... with Dynamic Dims", Wave February 2025 Release,
 *     FlashDecoding list), grouped-query heads, and a log-sum-exp combine of
 *     the splits (the split-KV grid and its empty-window handling follow the
 *     ideas of aiter PR 7412, Summary and Changes/Host side).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, dense
 *     (contiguous) in the layout named below, 16-byte aligned.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; 0 is the
 *     legacy default stream).  No entry point synchronizes the device.
 *   - Arguments are validated on the host before anything is launched; a bad
 *     argument returns ATTN_ERR_INVALID_ARG or ATTN_ERR_UNSUPPORTED and
 *     launches nothing.  attn_last_error() then describes the problem.
 *   - A launch failure returns ATTN_ERR_CUDA.
 *   - Kernels never spin without bound: every internal wait has a time limit
 *     after which the kernel records a device error word and exits;
 *     attn_device_error() reads it.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = -1,    /* a pointer, size or layout is invalid */
  ATTN_ERR_UNSUPPORTED = -2,    /* valid but not implemented (e.g. D not 64/128) */
  ATTN_ERR_CUDA = -3,           /* a CUDA runtime/driver call failed */
  ATTN_ERR_NO_MEMORY = -4,      /* workspace could not be (re)allocated */
  ATTN_ERR_DEVICE_TIMEOUT = -5  /* a kernel wait ran past its time limit */
} attn_status;

typedef enum { ATTN_BHSD = 0, ATTN_BSHD = 1 } attn_layout;

typedef enum { ATTN_F16 = 0, ATTN_BF16 = 1 } attn_dtype;

/*
 * Prefill attention forward.
 *
 * Defines: O[b,h,i,:] = sum_j softmax_j(scale * q_i . k_j) v_j over the keys j
 * visible to query i (WAVE MLSys 2026 summary, Attention (prefill)).
 *
 *   q   [B,H,S_q,D]  (layout ATTN_BHSD) or [B,S_q,H,D] (ATTN_BSHD), dtype
 *   k,v [B,H,S_kv,D] or [B,S_kv,H,D], same layout and dtype as q
 *   o   output, same shape, layout and dtype as q
 *   lse output [B,H,S_q] fp32, natural-log row sums ln sum_j exp(scale q.k_j);
 *       may be NULL.  A row with no visible key gets o = 0 and lse = -inf.
 *   causal  0 or 1.  Causal masking is bottom-right aligned: key j is visible
 *       to query i iff j <= i + (S_kv - S_q).
 *   scale   softmax scale, finite and > 0 (typically 1/sqrt(D)).
 *   D       64 or 128 (else ATTN_ERR_UNSUPPORTED).
 *   B, H, S_q, S_kv >= 0; B*H*S_q == 0 is a no-op.
 * Accumulation is fp32; P is rounded to the input dtype before P V; O is
 * rounded once, to nearest even.
 * The library keeps one int per (device, stream), created on the stream's
 * first call outside capture and zeroed on the stream before every launch:
 * persistent CTAs take their query blocks from it.  A call captured on a
 * stream that has none runs one CTA per query block (same results).  A
 * captured graph must not be replayed concurrently with other prefill work
 * of its capture stream (they share that counter).  attn_release_workspace
 * frees these counters too.
 */
ATTN_API attn_status attn_prefill_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int S_q, int S_kv, int D, attn_layout layout,
                             attn_dtype dtype, int causal, float scale, cudaStream_t stream);

/*
 * FP8 MQA logits (the indexer-style op of aiter PR 7412, "[FlyDSL] FP8 MQA
 * logits improvements for gfx950"; the page names its parts but prints no
 * formula, and this is the reading taken):
 *
 *   logits[i,j] = sum_h weights[i,h] * max(0, kv_scale[j] * (q[i,h] . kv[j]))
 *
 * for j in row i's window [window_start[i], window_end[i]) clamped to
 * [0, S_kv); outside it logits[i,j] = -inf if clean_logits, else untouched.
 *
 *   q             [S_q, H, D] E4M3 codes (torch.float8_e4m3fn)
 *   kv            [S_kv, D] E4M3 codes, one key row shared by every head
 *   kv_scale      [S_kv] fp32 per-key scale
 *   weights       [S_q, H] fp32
 *   window_start, [S_q] int32 on the device; any values (empty and
 *   window_end    past-the-end windows are fine)
 *   logits        [S_q, logits_stride] fp32 output, logits_stride >= S_kv
 *   H             32, 64 or 128; D = 128 (else ATTN_ERR_UNSUPPORTED).
 * Products are exact (E4M3 x E4M3) and accumulated in fp32.  Allocates
 * nothing.
 */
ATTN_API attn_status attn_mqa_logits_fp8(const void* q, const void* kv, const float* kv_scale,
                                         const float* weights, const int32_t* window_start,
                                         const int32_t* window_end, float* logits, int S_q,
                                         int S_kv, int H, int D, int64_t logits_stride,
                                         int clean_logits, cudaStream_t stream);

/*
 * Attention backward: gradients of attn_prefill_fwd's O.
 *
 * Defines, for the upstream gradient dO of O and P the softmax of the
 * forward ("Backward Flash Attention", Wave February 2025 Release, EvoFormer
 * list):  D_i = dO_i . O_i,  dS_ij = P_ij (dO_i . v_j - D_i),
 *         dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
 *         dV_j = sum_i P_ij dO_i  over the visible (i, j) pairs.
 *
 *   q, k, v, o  the forward's inputs and output (layout and dtype as there)
 *   dout        dO, q's shape, layout and dtype
 *   lse         [B,H,S_q] fp32, the lse the forward returned
 *   dq, dk, dv  outputs, the shapes of q, k, v, same layout and dtype
 *   delta       [B,H,S_q] fp32 scratch owned by the caller (overwritten with D)
 *   D           128 only (else ATTN_ERR_UNSUPPORTED); S_q, S_kv > 0; other
 *               arguments as for attn_prefill_fwd.
 * Deterministic: no atomics; P and dS are rounded to the input dtype before
 * their products, accumulation is fp32.  Allocates nothing.
 */
ATTN_API attn_status attn_prefill_bwd(const void* q, const void* k, const void* v, const void* o,
                                      const void* dout, const float* lse, void* dq, void* dk,
                                      void* dv, float* delta, int B, int H, int S_q, int S_kv,
                                      int D, attn_layout layout, attn_dtype dtype, int causal,
                                      float scale, cudaStream_t stream);

/*
 * FP8 prefill attention forward: the prefill operation on E4M3 inputs.
 *
 * Defines: attn_prefill_fwd's O and lse for Q = descale_q * q, K = descale_k *
 * k, V = descale_v * v, where q, k, v hold OCP 8-bit E4M3 codes (the layout
 * of torch.float8_e4m3fn) ("FAv3 - FP8", Wave February 2025 Release,
 * EvoFormer list).
 *
 *   q, k, v    E4M3 bytes, [B,H,S,D] (ATTN_BHSD) or [B,S,H,D] (ATTN_BSHD)
 *   o          output in out_dtype (ATTN_F16 or ATTN_BF16), q's shape and layout
 *   lse        [B,H,S_q] fp32 natural-log row sums of the real scores, or NULL
 *   descale_*  per-tensor factors, finite and > 0
 *   D          128 only (else ATTN_ERR_UNSUPPORTED); other arguments, and the
 *              per-stream unit counter, as for attn_prefill_fwd.
 * Both products run on E4M3 operands with fp32 accumulation; P is rounded to
 * E4M3 (relative error up to 2^-4 per weight) before P V, which sets the
 * accuracy: about 2-3% relative L2 error on O for N(0,1) inputs, independent
 * of the sequence length.
 */
ATTN_API attn_status attn_prefill_fp8_fwd(const void* q, const void* k, const void* v, void* o,
                                          float* lse, int B, int H, int S_q, int S_kv, int D,
                                          attn_layout layout, attn_dtype out_dtype, int causal,
                                          float scale, float descale_q, float descale_k,
                                          float descale_v, cudaStream_t stream);

/*
 * Extend attention forward: prefill of S_q new tokens per sequence against the
 * sequence's cached keys in a paged KV pool (prefix-cached / chunked prefill).
 *
 * Defines: O[b,i,h,:] = sum_t softmax_t(scale * q[b,i,h] . k_t) v_t over the
 * keys t < kv_lens[b] of sequence b visible to query i, read from kv head
 * g = h / (H_q / H_kv) ("Extend Attention", Wave February 2025 Release; the
 * SGLang extend mode, WAVE MLSys 2026 summary, Integration).  kv_lens[b]
 * counts the cached prefix AND the S_q new tokens, whose K/V the caller has
 * already written to the pool; with causal, key t is visible to query i iff
 * t <= i + (kv_lens[b] - S_q) (bottom-right, per sequence).
 *
 *   q          [B,S_q,H_q,D] dtype (BSHD)
 *   k_pool,    [num_pages, page_size, H_kv, D] dtype
 *   v_pool
 *   page_table [B, max_pages_per_seq] int32 pool page ids on the device;
 *              entries at or past ceil(kv_lens[b]/page_size) are never read,
 *              every entry read must be in [0, num_pages) (else the kernel
 *              reads zeros for that page and records device error code 2).
 *   kv_lens    [B] int32 on the device, 0 <= kv_lens[b] <= max_pages_per_seq *
 *              page_size (else clamped and device error code 2 recorded).  A
 *              query row with no visible key gets o = 0 and lse = -inf.
 *   o          [B,S_q,H_q,D] dtype output.
 *   lse        [B,H_q,S_q] fp32 natural-log row sums, or NULL.
 *   page_size  8, 16, 32, 64 or a multiple of 128 (else ATTN_ERR_UNSUPPORTED).
 *   H_q % H_kv == 0; D 64 or 128; causal 0 or 1; scale finite and > 0.
 *   B*S_q == 0 is a no-op.  Keys past kv_lens[b] in a page may hold any bit
 *   pattern, NaN included: they never reach the output.
 * Accumulation is fp32; P is rounded to the input dtype before P V.
 * Allocates nothing.
 */
ATTN_API attn_status attn_extend_fwd(const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* page_table, const int32_t* kv_lens, void* o,
                            float* lse, int B, int S_q, int H_q, int H_kv, int D, int page_size,
                            int max_pages_per_seq, int num_pages, attn_dtype dtype, int causal,
                            float scale, cudaStream_t stream);

/*
 * Decode attention forward (one query per head, split KV, paged or contiguous
 * KV cache).
 *
 * Defines: O[b,h,:] = sum_t softmax_t(scale * q[b,h] . k_t) v_t over the keys
 * t < kv_lens[b] of sequence b, read from kv head g = h / (H_q / H_kv)
 * (flash decoding, Wave February 2025 Release, FlashDecoding list).
 *
 *   q          [B,H_q,D] dtype
 *   k_pool,    paged: [num_pages, page_size, H_kv, D] dtype;
 *   v_pool     contiguous (page_table == NULL): [B, page_size, H_kv, D], i.e.
 *              page_size is the cache capacity S_max and sequence b owns page b
 *   page_table [B, max_pages_per_seq] int32 pool page ids, or NULL.  Entry
 *              [b, p] holds logical keys [p*page_size, (p+1)*page_size) of
 *              sequence b; entries at or past ceil(kv_lens[b]/page_size) are
 *              never read.  Every entry that is read must be in [0, num_pages).
 *   kv_lens    [B] int32 on the device, 0 <= kv_lens[b] <= max_pages_per_seq *
 *              page_size.  A sequence with kv_len 0 gets o = 0.
 *   o          [B,H_q,D] dtype output.
 *   page_size  keys per page: when paged, 8, 16, 32 or a multiple of 64 (else
 *              ATTN_ERR_UNSUPPORTED); when contiguous, the capacity S_max (> 0).
 *   max_pages_per_seq  page_table row stride (ADDED to the published
 *              signature: the table's shape is not otherwise known); 1 when
 *              contiguous.
 *   num_pages  number of pages in the pool (ADDED: bounds the gather); B when
 *              contiguous.
 *   num_splits 0: split count chosen per sequence from its kv_len on the
 *              device; > 0: every sequence is split into that many parts.
 *   scale      softmax scale, finite and > 0.
 *   dtype      ATTN_F16 or ATTN_BF16 (ADDED: not in the published signature).
 *   H_q % H_kv == 0, H_q / H_kv <= 16, D 64 or 128 (else ATTN_ERR_UNSUPPORTED).
 * The library owns a split-partials workspace per (device, stream), grown on
 * demand outside stream capture; growing it during capture returns
 * ATTN_ERR_NO_MEMORY (call once with the largest shapes, on the stream that
 * will be captured, before capturing).  A graph captured from a call keeps
 * the workspace address of that call: a later call that has to grow the
 * workspace retires the old buffer without freeing it, so such graphs stay
 * valid until attn_release_workspace, which frees every buffer (after it,
 * graphs captured earlier must not be replayed).
 * Calls on different streams may run concurrently; calls on one stream use
 * its workspace in stream order.
 */
ATTN_API attn_status attn_decode_fwd(const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* page_table, const int32_t* kv_lens, void* o, int B,
                            int H_q, int H_kv, int D, int page_size, int max_pages_per_seq,
                            int num_pages, int num_splits, float scale, attn_dtype dtype,
                            cudaStream_t stream);

/*
 * Decode attention that allocates no device memory.  The source pages have no
 * counterpart: they never discuss who owns a kernel's workspace.
 *
 * Same arguments, rules and results as attn_decode_fwd (bitwise: the same
 * checks, split plan and kernels), for callers that cannot let a library
 * allocate: engines whose framework owns all device memory through its own
 * pool and budget, and serving loops that must not block on the allocator or
 * meet an out-of-memory error at step time.  The split partials live in one
 * fixed 16 MiB device array inside the library (held on every GPU that loads
 * it until the process exits) instead of a cudaMalloc'd workspace.  A call
 * whose split plan needs more (B * H_q * splits * (D + 1) * 4 bytes) returns
 * ATTN_ERR_UNSUPPORTED and launches nothing: pass num_splits > 0 with fewer
 * splits, or use attn_decode_fwd.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress); make that first call before
 * any stream capture.  All calls share the array and it keeps the last call's
 * contents (nothing in it needs to start at zero); calls whose kernels overlap
 * on the GPU race on it.
 */
ATTN_API attn_status attn_decode_fwd_noalloc(const void* q, const void* k_pool,
                                             const void* v_pool, const int32_t* page_table,
                                             const int32_t* kv_lens, void* o, int B, int H_q,
                                             int H_kv, int D, int page_size,
                                             int max_pages_per_seq, int num_pages,
                                             int num_splits, float scale, attn_dtype dtype,
                                             cudaStream_t stream);

/* Message describing the last error returned on the calling thread. */
ATTN_API const char* attn_last_error(void);

/*
 * Read (and clear, if `clear` != 0) the device error word of the current
 * device: 0 when no kernel recorded an error, else (code << 16) | site, where
 * code 1 = a wait ran past its time limit and code 2 = a kernel met an
 * argument it cannot use (a kv_len outside the page table's capacity, a page
 * id outside the pool).  Synchronizes the device first.
 * Returns ATTN_OK, or ATTN_ERR_DEVICE_TIMEOUT when the word was non-zero.
 */
ATTN_API attn_status attn_device_error(int* word, int clear);

/*
 * Set the time limit (nanoseconds) every kernel wait is bounded by; 0 restores
 * the default (4 s, or the ATTN_WAIT_LIMIT_NS environment variable if set when
 * the library was loaded).  Applies to launches made after the call.
 */
ATTN_API void attn_set_wait_limit_ns(uint64_t ns);

/*
 * Failure-detection self-test: launches one thread that waits, with the same
 * bounded wait every kernel uses, on an mbarrier nothing ever completes.
 * After limit_ns (0 < limit_ns <= 1e10) the wait gives up and records
 * (1 << 16) | 900 (a timed-out wait at site 900) in the device error word,
 * which attn_device_error() then reports; the context stays usable.
 * Returns ATTN_ERR_INVALID_ARG for a limit out of range.
 */
ATTN_API attn_status attn_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream);

/* Free the decode workspaces (current and retired) and prefill unit counters
 * of all streams of the current device; synchronizes the device (not during
 * capture).  CUDA graphs captured from earlier decode or prefill calls hold
 * those addresses and must not be replayed after it. */
ATTN_API attn_status attn_release_workspace(void);

/* Library version string. */
ATTN_API const char* attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
