// decode_sm103a.cu -- seq_len = 1 flash decoding for sm_103a: split-KV over a
// paged or contiguous KV cache, grouped-query heads, and a log-sum-exp combine.
//
// The method is the pages' "Flash Decoding Kernel" with and without paged
// attention and with dynamic (runtime) lengths (Wave February 2025 Release,
// FlashDecoding list); sequences are split along the KV axis (the split-KV
// grid of aiter PR 7412, Summary), empty splits are a no-op that the combine
// skips instead of widening any scan window (aiter PR 7412, Motivation and
// "Empty-window fix"), and the gather reads pages through a page table
// ("buffer loads ... gather", "dynamic symbols", Wave February 2025 Release).
//
// Blackwell design:
//  * grid = (split, kv head, batch); one CTA reads each K/V row of its key
//    range exactly once for all H_q/H_kv query heads of the group;
//  * a TMA warp gathers 64-key tiles of K and V (one tensor-map box per page
//    and 64-column half, 128-byte swizzle) into a 3-stage shared-memory ring;
//  * four consumer warps each take 16 keys of every tile: S = Q K^T and
//    O += P V with mma.sync m16n8k16 (the query group is 16 rows, far below
//    tcgen05's minimum, and the kernel is bound by HBM bandwidth), online
//    softmax in fp32, then the warps merge in shared memory;
//  * keys at or past the split end are masked to -inf and their V rows are
//    zeroed in shared memory, so page tails are never used even if they hold
//    non-finite garbage.
// Partials (normalised o and log2-sum-exp per split) go to a workspace that
// decode_combine_kernel reduces.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_sm103a.h"
#include "host_once.h"
#include "sm103a_ptx.cuh"

namespace attn_sm103a {

namespace {

constexpr int kKeysPerTile = 64;
constexpr int kConsumerWarps = 4;
constexpr int kKeysPerWarp = kKeysPerTile / kConsumerWarps;  // 16
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 3;

template <int D>
struct DCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kKeysPerTile * 128;           // 64 keys x 64 columns
  static constexpr int kTileBytes = kHalves * kHalfBytes;          // K (or V) of one tile
  static constexpr int kStageBytes = 2 * kTileBytes;               // K + V
  static constexpr int kRedBytes = kConsumerWarps * (32 + 16 * D) * 4;
  static constexpr int kSmemData = kStages * kStageBytes;
  static_assert(kRedBytes <= kSmemData, "reduction buffer must fit in the ring");
  static constexpr int kSmemBytes = kSmemData + 1024 + 128;
};

// Keys per split of a sequence of length kv.
__device__ __forceinline__ int split_chunk(int kv, const DecodeParams& p) {
  if (p.fixed_chunk > 0) return p.fixed_chunk;
  int c = (kv + p.num_splits - 1) / p.num_splits;
  c = (c + kKeysPerTile - 1) / kKeysPerTile * kKeysPerTile;
  return c < kKeysPerTile ? kKeysPerTile : c;
}

__device__ __forceinline__ int clamp_kv(int kv, const DecodeParams& p) {
  const int cap = p.max_pages * p.page_size;
  if (kv < 0 || kv > cap) {
    record_error(p.err, kErrBadArgument, 1);
    kv = kv < 0 ? 0 : cap;
  }
  return kv;
}

// Byte offset, inside one K or V tile, of the 16-byte chunk holding columns
// [8*chunk, 8*chunk+8) of 64-column half `half` of key `key` (TMA 128-byte
// swizzle: chunk index XOR row index mod 8).
__device__ __forceinline__ uint32_t tile_off(int key, int half, int chunk) {
  return static_cast<uint32_t>(half * (kKeysPerTile * 128) + key * 128 + ((chunk ^ (key & 7)) << 4));
}

template <int D, bool kBF16>
__global__ void __launch_bounds__(kThreads, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  using C = DCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kSmemData);
  uint64_t* empty = full + kStages;

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = p.group;
  const int kv = clamp_kv(p.kv_lens[b], p);
  const int chunk = split_chunk(kv, p);
  const int start = split * chunk;
  const int end = min(kv, start + chunk);
  const size_t part_row = (static_cast<size_t>(b) * p.H_q + static_cast<size_t>(g) * G);

  if (start >= end) {  // empty split: contributes nothing to the combine
    if (threadIdx.x < G) p.lse_part[(part_row + threadIdx.x) * p.max_splits + split] = -INFINITY;
    return;
  }
  const int n_tiles = (end - start + kKeysPerTile - 1) / kKeysPerTile;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------- producer
    // The whole warp runs the loop: it keeps a window of 32 page ids in
    // registers (lane l holds entry window_base + l, refilled with one
    // coalesced load) and each lane issues one TMA box of the tile, so a
    // tile costs one instruction issue instead of a dependent page-table
    // load per page.
    if (lane == 0) {
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
    }
    const bool paged = p.page_table != nullptr;
    const int ps = p.page_size;
    const int box_rows = paged ? min(ps, kKeysPerTile) : kKeysPerTile;
    const int boxes_per_tile = paged ? kKeysPerTile / box_rows : 1;
    const int32_t* pt = paged ? p.page_table + static_cast<size_t>(b) * p.max_pages : nullptr;
    const int n_pages_seq = paged ? (kv + ps - 1) / ps : 0;  // entries that may be read
    int window_base = -(1 << 30);
    int window_page = 0;
    int issued = 0;
    for (int it = 0; it < n_tiles; ++it) {
      const int st = it % kStages;
      const int round = it / kStages;
      if (round > 0) {
        const bool ok = mbar_wait(&empty[st], (round - 1) & 1, p.wait_limit_ns, p.err, 50);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      const int k0 = start + it * kKeysPerTile;
      const int n_box = paged ? min(boxes_per_tile, (end - k0 + box_rows - 1) / box_rows) : 1;
      int page = b, slot = 0;
      const int bx = lane / (2 * C::kHalves);
      if (paged) {
        const int first_p = k0 / ps;
        const int last_p = (min(k0 + kKeysPerTile, end) - 1) / ps;
        if (last_p >= window_base + 32) {  // refill (pages only move forward)
          window_base = first_p;
          const int e = window_base + lane;
          window_page = e < n_pages_seq ? pt[e] : 0;
        }
        const int key = k0 + min(bx, n_box - 1) * box_rows;
        page = __shfl_sync(0xffffffffu, window_page, key / ps - window_base);
        slot = key % ps;
        if (page < 0 || page >= p.num_pages) {  // the TMA would zero-fill; flag it
          if (bx < n_box) record_error(p.err, kErrBadArgument, 2);
          page = p.num_pages;
        }
      } else {
        slot = k0;
      }
      if (lane == 0)
        mbar_arrive_expect_tx(&full[st], 2 * C::kHalves * n_box * box_rows * 128);
      __syncwarp();
      if (bx < n_box) {
        const int hf = (lane / 2) % C::kHalves;
        const bool is_v = lane & 1;
        uint8_t* dst = smem + st * C::kStageBytes + (is_v ? C::kTileBytes : 0) +
                       hf * C::kHalfBytes + bx * box_rows * 128;
        tma_load_4d(dst, is_v ? &tm_v : &tm_k, &full[st], hf * 64, g, slot, page);
      }
      issued = it + 1;
    }
    if (lane == 0)
      for (int it = max(0, issued - kStages); it < issued; ++it)
        mbar_wait(&full[it % kStages], (it / kStages) & 1, p.wait_limit_ns, p.err, 51);
    __syncwarp();
    return;  // the producer takes no part in the final merge
  }

  // --------------------------------------------------------------- consumers
  const int r0 = lane / 4, r1 = lane / 4 + 8;  // fragment rows (query heads)
  const int cq = 2 * (lane % 4);                // fragment column pair
  const float c = p.scale_log2;

  // Q fragments (A operand, rows = heads of the group, zero past G).
  uint32_t qa[D / 16][4];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q);
    const size_t row0 = (part_row + r0) * (D / 2), row1 = (part_row + r1) * (D / 2);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int cidx = (ks * 16 + cq) / 2;
      qa[ks][0] = r0 < G ? q32[row0 + cidx] : 0u;
      qa[ks][1] = r1 < G ? q32[row1 + cidx] : 0u;
      qa[ks][2] = r0 < G ? q32[row0 + cidx + 4] : 0u;
      qa[ks][3] = r1 < G ? q32[row1 + cidx + 4] : 0u;
    }
  }

  float m[2] = {-INFINITY, -INFINITY};
  float l[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;

  const int wkey = warp * kKeysPerWarp;  // this warp's first key in each tile
  bool ok = true;
  for (int it = 0; it < n_tiles; ++it) {
    const int st = it % kStages;
    ok = __all_sync(0xffffffffu,
                    mbar_wait(&full[st], (it / kStages) & 1, p.wait_limit_ns, p.err, 52));
    if (!ok) break;
    uint8_t* kd = smem + st * C::kStageBytes;
    uint8_t* vd = kd + C::kTileBytes;
    const int k0 = start + it * kKeysPerTile + wkey;  // logical key of this warp's row 0
    if (k0 < end) {
      if (k0 + kKeysPerWarp > end) {
        // Zero this warp's V rows at or past the split end (page tails).
        for (int e = lane; e < kKeysPerWarp * C::kHalves * 8; e += 32) {
          const int kr = e / (C::kHalves * 8);
          const int hf = (e / 8) % C::kHalves;
          if (k0 + kr >= end)
            *reinterpret_cast<uint4*>(vd + tile_off(wkey + kr, hf, e % 8)) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      // S = Q K^T for 16 keys: two n-tiles of 8 keys.
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const uint32_t kbase = smem_u32(kd);
      const int mi = lane / 8, mr = lane % 8;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t bf[4];
        const int key = wkey + (mi / 2) * 8 + mr;
        const int col = (ks % 4) * 2 + (mi % 2);
        ldsm_x4(kbase + tile_off(key, ks / 4, col), bf);
        mma_16816<kBF16>(sacc[0], qa[ks], bf[0], bf[1]);
        mma_16816<kBF16>(sacc[1], qa[ks], bf[2], bf[3]);
      }
      // Scale, mask, online softmax (rows r0: elements 0,1; r1: elements 2,3).
      float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = k0 + nt * 8 + cq + (e & 1);
          const float v = key < end ? sacc[nt][e] * c : -INFINITY;
          sacc[nt][e] = v;
          mt[e / 2] = fmaxf(mt[e / 2], v);
        }
      float alpha[2], mref[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        mt[rr] = fmaxf(mt[rr], __shfl_xor_sync(0xffffffffu, mt[rr], 1));
        mt[rr] = fmaxf(mt[rr], __shfl_xor_sync(0xffffffffu, mt[rr], 2));
        const float m_new = fmaxf(m[rr], mt[rr]);
        alpha[rr] = (m_new == -INFINITY) ? 1.f : ex2_approx(m[rr] - m_new);
        mref[rr] = (m_new == -INFINITY) ? 0.f : m_new;
        m[rr] = m_new;
      }
      float rs[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float pv = ex2_approx(sacc[nt][e] - mref[e / 2]);
          sacc[nt][e] = pv;
          rs[e / 2] += pv;
        }
      l[0] = l[0] * alpha[0] + rs[0];
      l[1] = l[1] * alpha[1] + rs[1];
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        o[dn][0] *= alpha[0];
        o[dn][1] *= alpha[0];
        o[dn][2] *= alpha[1];
        o[dn][3] *= alpha[1];
      }
      uint32_t pa[4];
      pa[0] = pack2<kBF16>(sacc[0][0], sacc[0][1]);
      pa[1] = pack2<kBF16>(sacc[0][2], sacc[0][3]);
      pa[2] = pack2<kBF16>(sacc[1][0], sacc[1][1]);
      pa[3] = pack2<kBF16>(sacc[1][2], sacc[1][3]);
      // O += P V: V^T fragments by transposed ldmatrix, two 8-column n-tiles each.
      const uint32_t vbase = smem_u32(vd);
#pragma unroll
      for (int dn = 0; dn < D / 8; dn += 2) {
        uint32_t bf[4];
        const int key = wkey + (mi % 2) * 8 + mr;
        const int col0 = (dn + mi / 2) * 8;  // first column of this 8x8 block
        ldsm_x4_trans(vbase + tile_off(key, col0 / 64, (col0 % 64) / 8), bf);
        mma_16816<kBF16>(o[dn], pa, bf[0], bf[1]);
        mma_16816<kBF16>(o[dn + 1], pa, bf[2], bf[3]);
      }
    }
    fence_proxy_async_smem();  // our zeroing writes precede the next TMA into this stage
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // Row sums over the 4 lanes that share a row.
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 1);
    l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 2);
  }

  // ----------------------------------------------------- merge the 4 warps
  named_barrier_sync(1, kConsumerWarps * 32);  // every warp is done with the ring
  float* red = reinterpret_cast<float*>(smem);
  float* red_w = red + warp * (32 + 16 * D);   // [m 16][l 16][o 16 x D]
  if (lane % 4 == 0) {
    red_w[r0] = ok ? m[0] : -INFINITY;
    red_w[r1] = ok ? m[1] : -INFINITY;
    red_w[16 + r0] = l[0];
    red_w[16 + r1] = l[1];
  }
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) {
    const int col = dn * 8 + cq;
    red_w[32 + r0 * D + col] = o[dn][0];
    red_w[32 + r0 * D + col + 1] = o[dn][1];
    red_w[32 + r1 * D + col] = o[dn][2];
    red_w[32 + r1 * D + col + 1] = o[dn][3];
  }
  named_barrier_sync(1, kConsumerWarps * 32);
  for (int idx = threadIdx.x; idx < G * D; idx += kConsumerWarps * 32) {
    const int r = idx / D, d = idx % D;
    float mw[kConsumerWarps];
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      mw[w] = red[w * (32 + 16 * D) + r];
      M = fmaxf(M, mw[w]);
    }
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float* rw = red + w * (32 + 16 * D);
      const float sc = (mw[w] == -INFINITY) ? 0.f : ex2_approx(mw[w] - M);
      L += sc * rw[16 + r];
      O += sc * rw[32 + r * D + d];
    }
    const size_t prow = (part_row + r) * p.max_splits + split;
    p.o_part[prow * D + d] = (L > 0.f) ? O / L : 0.f;
    if (d == 0) p.lse_part[prow] = (L > 0.f) ? M + __log2f(L) : -INFINITY;
  }
}

// One CTA per (query head, batch): O = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M).
template <int D, bool kBF16>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodeParams p, void* out) {
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int kv = clamp_kv(p.kv_lens[b], p);
  const int chunk = split_chunk(kv, p);
  const int n = kv > 0 ? min(p.max_splits, (kv + chunk - 1) / chunk) : 0;
  const size_t row = (static_cast<size_t>(b) * p.H_q + h) * p.max_splits;
  float M = -INFINITY;
  for (int s = 0; s < n; ++s) M = fmaxf(M, p.lse_part[row + s]);
  float L = 0.f, O = 0.f;
  for (int s = 0; s < n; ++s) {
    const float ls = p.lse_part[row + s];
    if (ls == -INFINITY) continue;
    const float w = ex2_approx(ls - M);
    L += w;
    O += w * p.o_part[(row + s) * D + d];
  }
  const float val = L > 0.f ? O / L : 0.f;
  const size_t oi = (static_cast<size_t>(b) * p.H_q + h) * D + d;
  if constexpr (kBF16)
    reinterpret_cast<__nv_bfloat16*>(out)[oi] = __float2bfloat16_rn(val);
  else
    reinterpret_cast<__half*>(out)[oi] = __float2half_rn(val);
}

template <int D, bool kBF16>
cudaError_t launch_decode_t(const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p,
                            void* out, cudaStream_t stream) {
  auto kern = decode_split_kernel<D, kBF16>;
  static std::atomic<unsigned long long> configured{0};  // per template instance, per device
  cudaError_t ce = attn_host::once_per_device(configured, [&]() {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                DCfg<D>::kSmemBytes);
  });
  if (ce != cudaSuccess) return ce;
  dim3 grid(p.max_splits, p.H_q / p.group, p.B);
  kern<<<grid, kThreads, DCfg<D>::kSmemBytes, stream>>>(k, v, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<D, kBF16><<<dim3(p.H_q, p.B), D, 0, stream>>>(p, out);
  return cudaGetLastError();
}

}  // namespace

cudaError_t decode_launch(const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p,
                          void* out, int D, bool bf16, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  if (D == 128) return bf16 ? launch_decode_t<128, true>(k, v, p, out, stream)
                            : launch_decode_t<128, false>(k, v, p, out, stream);
  return bf16 ? launch_decode_t<64, true>(k, v, p, out, stream)
              : launch_decode_t<64, false>(k, v, p, out, stream);
}

int decode_keys_per_tile() { return kKeysPerTile; }

}  // namespace attn_sm103a
