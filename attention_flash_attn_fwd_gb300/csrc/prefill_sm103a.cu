// prefill_sm103a.cu -- fused attention forward (prefill form) for sm_103a.
//
//   O = softmax(scale * Q K^T + causal mask) V,   lse = ln sum_j exp(scale q.k_j)
//
// The operation is the one the pages call "attention" / "prefill attention"
// (WAVE MLSys 2026 summary, Attention (prefill), Figures 2-4; Wave February
// 2025 Release, "Prefill attention kernel"), over BHSD or BSHD tensors (the
// same computation with the sequence and head strides swapped, WAVE summary,
// Assumption 1).  The pages' own kernels are AMD MFMA/LDS designs; this one
// is written for Blackwell:
//
//  * one CTA owns 256 query rows of one (batch, head) as two 128-row tiles;
//  * a TMA warp streams K_j and V_j (128 keys each) through a ring of
//    128-byte-swizzled shared-memory stages (multi-buffering, Wave February
//    2025 Release, Multi-Buffering; global-read coarsening, WAVE summary
//    section 4, becomes whole-tile TMA copies);
//  * an MMA warp issues tcgen05.mma: S_t = Q_t K_j^T into tensor memory, then
//    O_t += P_t V_j with P_t read straight from tensor memory;
//  * two softmax warpgroups, one per query tile, alternate (the two tiles
//    ping-pong so one tile's softmax overlaps the other's MMAs; "subgroup
//    ping-pong", WAVE summary, Schedule reordering): each thread owns one
//    query row, keeps its running max and sum in fp32, writes P over S in
//    tensor memory, and rescales O only when the row max grew by more than
//    2^8 (the exact result is unchanged: O and l always share one reference);
//  * causal tiles wholly above the diagonal are never loaded or multiplied
//    (tile skipping, aiter PR 7412, Changes/Kernel "tile_skip"), only the
//    diagonal tiles are masked element by element.
//
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D),
// O1 [256+D, 256+2D).  P_t (16-bit pairs) overwrites the first 64 columns of
// S_t.
#include "prefill_sm103a.h"
#include "sm103a_ptx.cuh"

namespace attn_sm103a {

namespace {

constexpr int kBM = 128;      // query rows per tile
constexpr int kBN = 128;      // keys per KV tile
constexpr int kTiles = 2;     // query tiles per CTA
constexpr int kThreads = 320; // 8 softmax warps + TMA warp + MMA warp
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Cfg {
  static constexpr int kTileBytes = kBM * D * 2;          // one Q/K/V/O tile
  static constexpr int kStages = (D == 128) ? 4 : 8;      // KV ring depth
  static constexpr int kSmemData = kTiles * kTileBytes + kStages * kTileBytes;
  static constexpr int kSmemBytes = kSmemData + 1024 /*align*/ + 256 /*barriers*/;
  // tensor-memory columns of S_t and O_t
  __device__ static constexpr uint32_t col_s(int t) { return t * 128u; }
  __device__ static constexpr uint32_t col_o(int t) { return 256u + t * D; }
};

struct SharedCtl {
  uint64_t q_full[kTiles];
  uint64_t s_full[kTiles];
  uint64_t p_full[kTiles];
  uint64_t o_full;
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint32_t tmem_base;
  int abort;
};

// TMA load of one 64-column box of rows [row, row + 128) of (batch b, head h).
// BHSD maps are (D, S, H, B); BSHD maps are (D, H, S, B).
__device__ __forceinline__ void load_box(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                         int row, int h, int b, int bshd) {
  if (bshd)
    tma_load_4d(dst, map, bar, x, h, row, b);
  else
    tma_load_4d(dst, map, bar, x, row, h, b);
}

// Number of KV tiles a query tile [row0, row0 + kBM) must visit.
__device__ __forceinline__ int kv_tiles_for(int row0, const PrefillParams& p) {
  int keys = p.S_kv;
  if (p.causal) {
    int last_row = min(row0 + kBM, p.S_q) - 1;
    keys = min(keys, last_row + (p.S_kv - p.S_q) + 1);
  }
  return keys <= 0 ? 0 : (keys + kBN - 1) / kBN;
}

template <int D, bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o, const PrefillParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* s_q = smem;                                   // kTiles tiles
  uint8_t* s_kv = smem + kTiles * C::kTileBytes;         // kStages tiles
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + C::kSmemData);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // Work item: (batch, head, 256-row query block); the longest causal blocks
  // of a (batch, head) are handed out first, heads stay adjacent for L2 reuse.
  const int nqb = p.num_q_blocks;
  const int bh = blockIdx.x / nqb;
  const int qb = nqb - 1 - (blockIdx.x % nqb);
  const int b = bh / p.H;
  const int h = bh % p.H;
  const int row_base = qb * (kTiles * kBM);
  int n_kv[kTiles];
#pragma unroll
  for (int t = 0; t < kTiles; ++t) n_kv[t] = kv_tiles_for(row_base + t * kBM, p);
  const int n_all = max(n_kv[0], n_kv[1]);  // tile 1 never needs fewer than tile 0

  if (warp == kWarpMma) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&ctl->q_full[t], 1);
      mbar_init(&ctl->s_full[t], 1);
      mbar_init(&ctl->p_full[t], 4);
    }
    mbar_init(&ctl->o_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&ctl->kv_full[s], 1);
      mbar_init(&ctl->kv_empty[s], 1);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_all > 0) {
      int issued = 0;  // KV loads issued so far
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      for (int t = 0; t < kTiles; ++t) {
        mbar_arrive_expect_tx(&ctl->q_full[t], C::kTileBytes);
        for (int x = 0; x < D / 64; ++x)
          load_box(s_q + t * C::kTileBytes + x * (kBM * 128), &tm_q, &ctl->q_full[t], x * 64,
                   row_base + t * kBM, h, b, p.bshd);
      }
      volatile int* abort_flag = &ctl->abort;
      for (int j = 0; j < n_all && !*abort_flag; ++j) {
#pragma unroll
        for (int kind = 0; kind < 2; ++kind) {
          const int idx = 2 * j + kind;
          const int st = idx % C::kStages;
          const int round = idx / C::kStages;
          if (round > 0 &&
              !mbar_wait(&ctl->kv_empty[st], (round - 1) & 1, p.wait_limit_ns, p.err, 10)) {
            *abort_flag = 1;
            break;
          }
          uint8_t* dst = s_kv + st * C::kTileBytes;
          mbar_arrive_expect_tx(&ctl->kv_full[st], C::kTileBytes);
          const CUtensorMap* map = kind == 0 ? &tm_k : &tm_v;
          for (int x = 0; x < D / 64; ++x)
            load_box(dst + x * (kBN * 128), map, &ctl->kv_full[st], x * 64, j * kBN, h, b,
                     p.bshd);
          issued = idx + 1;
        }
      }
      // Never leave the CTA with a copy still landing in shared memory: wait
      // (bounded) for the last load issued into every stage and for Q.
      for (int idx = max(0, issued - C::kStages); idx < issued; ++idx)
        mbar_wait(&ctl->kv_full[idx % C::kStages], (idx / C::kStages) & 1, p.wait_limit_ns,
                  p.err, 11);
      for (int t = 0; t < kTiles; ++t) mbar_wait(&ctl->q_full[t], 0, p.wait_limit_ns, p.err, 12);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_all > 0) {
      constexpr uint32_t id_s = idesc_f16(kBF16, kBM, kBN, false, false);
      constexpr uint32_t id_o = idesc_f16(kBF16, kBM, D, false, true);
      const uint32_t q_addr = smem_u32(s_q);
      const uint32_t kv_addr = smem_u32(s_kv);
      bool ok = true;
      for (int t = 0; t < kTiles && ok; ++t)
        ok = mbar_wait(&ctl->q_full[t], 0, p.wait_limit_ns, p.err, 20);

      // S_t = Q_t K_j^T  (both operands K-major, 128-byte swizzle)
      auto issue_s = [&](int t, int st) {
        const uint32_t qa = q_addr + t * C::kTileBytes;
        const uint32_t ka = kv_addr + st * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * (kBM * 128) + (kk % 4) * 32;
          mma_ss(tmem + C::col_s(t), sdesc_sw128(qa + off, 16, 1024),
                 sdesc_sw128(ka + off, 16, 1024), id_s, kk > 0);
        }
      };
      // O_t (+)= P_t V_j  (P from tensor memory, V MN-major, 128-byte swizzle)
      auto issue_pv = [&](int t, int st, bool acc) {
        const uint32_t va = kv_addr + st * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(tmem + C::col_o(t), tmem + C::col_s(t) + kk * 8,
                 sdesc_sw128(va + kk * 16 * 128, kBN * 128, 1024), id_o,
                 (acc || kk > 0) ? 1u : 0u);
      };
      auto wait_full = [&](int idx, int site) {
        return mbar_wait(&ctl->kv_full[idx % C::kStages], (idx / C::kStages) & 1,
                         p.wait_limit_ns, p.err, site);
      };

      if (ok && (ok = wait_full(0, 21))) {
        tc_fence_after_sync();
        for (int t = 0; t < kTiles; ++t)
          if (n_kv[t] > 0) {
            issue_s(t, 0);
            mma_commit(&ctl->s_full[t]);
          }
        mma_commit(&ctl->kv_empty[0]);
      }
      for (int j = 0; j < n_all && ok; ++j) {
        const int st_v = (2 * j + 1) % C::kStages;
        const int st_kn = (2 * j + 2) % C::kStages;
        const bool next = j + 1 < n_all;
        bool kn_ready = false;
        if (!(ok = wait_full(2 * j + 1, 22))) break;
        for (int t = 0; t < kTiles && ok; ++t) {
          if (j < n_kv[t]) {
            if (!(ok = mbar_wait(&ctl->p_full[t], j & 1, p.wait_limit_ns, p.err, 23 + t))) break;
            tc_fence_after_sync();
            issue_pv(t, st_v, j > 0);
          }
          if (t == kTiles - 1) mma_commit(&ctl->kv_empty[st_v]);
          if (next) {
            if (!kn_ready) {
              if (!(ok = wait_full(2 * j + 2, 25))) break;
              kn_ready = true;
              tc_fence_after_sync();
            }
            if (j + 1 < n_kv[t]) {
              issue_s(t, st_kn);
              mma_commit(&ctl->s_full[t]);
            }
            if (t == kTiles - 1) mma_commit(&ctl->kv_empty[st_kn]);
          }
        }
      }
      mma_commit(&ctl->o_full);
      if (!ok) *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
      // No MMA may still be running when tensor memory is released.
      mbar_wait(&ctl->o_full, 0, p.wait_limit_ns, p.err, 26);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp / 4;             // query tile of this warpgroup
    const int wl = warp % 4;            // warp's TMEM lane quarter
    const int r = wl * 32 + lane;       // row within the tile
    const int row0 = row_base + t * kBM;
    const int i = row0 + r;             // query index
    const int diag = p.S_kv - p.S_q;    // bottom-right causal offset
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wl * 32) << 16);
    const uint32_t col_s = C::col_s(t);
    const uint32_t col_o = C::col_o(t);
    const float c = p.scale_log2;

    float m2 = -INFINITY;  // running reference max, scaled log2 units
    float l = 0.f;         // running sum of exponentials relative to m2
    bool ok = true;
    for (int j = 0; j < n_kv[t]; ++j) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&ctl->s_full[t], j & 1, p.wait_limit_ns, p.err, 30 + t));
      if (!ok) break;
      tc_fence_after_sync();
      float s[kBN];
      tmem_ld64_wait(lane_addr + col_s, *reinterpret_cast<float(*)[64]>(&s[0]));
      tmem_ld64_wait(lane_addr + col_s + 64, *reinterpret_cast<float(*)[64]>(&s[64]));
      const int key0 = j * kBN;
      const bool full = (key0 + kBN <= p.S_kv) && (!p.causal || key0 + kBN - 1 <= row0 + diag);
      if (!full) {
        const int lim = p.causal ? min(p.S_kv - 1, i + diag) : p.S_kv - 1;
#pragma unroll
        for (int cc = 0; cc < kBN; ++cc)
          if (key0 + cc > lim) s[cc] = -INFINITY;
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int cc = 4; cc < kBN; cc += 4) {
        mx0 = fmaxf(mx0, s[cc]);
        mx1 = fmaxf(mx1, s[cc + 1]);
        mx2 = fmaxf(mx2, s[cc + 2]);
        mx3 = fmaxf(mx3, s[cc + 3]);
      }
      const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
      const float m_new = fmaxf(m2, m_tile);
      float alpha = 1.f;
      bool need = false;
      if (m_new > m2 + kRescaleThreshold) {  // false while m_new == -inf
        alpha = ex2_approx(m2 - m_new);      // 0 on the first visible tile
        need = (j > 0);
        m2 = m_new;
      }
      const float mref = (m2 == -INFINITY) ? 0.f : m2;
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const float e0 = ex2_approx(fmaf(s[half * 64 + 2 * q], c, -mref));
          const float e1 = ex2_approx(fmaf(s[half * 64 + 2 * q + 1], c, -mref));
          sum0 += e0;
          sum1 += e1;
          pk[q] = pack2<kBF16>(e0, e1);
        }
        tmem_st32(lane_addr + col_s + half * 32, pk);
      }
      l = l * alpha + (sum0 + sum1);
      if (__any_sync(0xffffffffu, need)) {
        // O_t row *= alpha.  PV_t,j-1 completed before S_t,j was signalled.
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld32_wait(lane_addr + col_o + cc, o);
#pragma unroll
          for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
          tmem_st32(lane_addr + col_o + cc, o);
        }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->p_full[t]);
    }

    // ------------------------------------------------------------ epilogue
    if (ok && n_all > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->o_full, 0, p.wait_limit_ns, p.err, 40 + t));
    tc_fence_after_sync();
    const bool have_o = ok && n_kv[t] > 0 && l > 0.f;
    const float inv_l = have_o ? 1.f / l : 0.f;
    uint8_t* s_o = s_q + t * C::kTileBytes;  // Q_t is dead once o_full fired
#pragma unroll 1
    for (int cc = 0; cc < D; cc += 64) {
      uint32_t o[64] = {};
      if (n_kv[t] > 0 && ok) tmem_ld64_wait(lane_addr + col_o + cc, o);
      uint8_t* sub = s_o + (cc / 64) * (kBM * 128) + r * 128;
#pragma unroll
      for (int q = 0; q < 8; ++q) {  // 8 chunks of 8 columns = 16 bytes each
        uint4 w;
        uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float v0 = have_o ? __uint_as_float(o[q * 8 + 2 * e]) * inv_l : 0.f;
          const float v1 = have_o ? __uint_as_float(o[q * 8 + 2 * e + 1]) * inv_l : 0.f;
          wp[e] = pack2<kBF16>(v0, v1);
        }
        *reinterpret_cast<uint4*>(sub + ((q ^ (r & 7)) * 16)) = w;
      }
    }
    if (p.lse != nullptr && i < p.S_q) {
      const float lse = have_o ? (m2 + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      p.lse[(static_cast<size_t>(b) * p.H + h) * p.S_q + i] = lse;
    }
    fence_proxy_async_smem();
    named_barrier_sync(1 + t, 128);
    if (wl == 0 && lane == 0 && row0 < p.S_q) {
      for (int x = 0; x < D / 64; ++x)
        if (p.bshd)
          tma_store_4d(&tm_o, s_o + x * (kBM * 128), x * 64, h, row0, b);
        else
          tma_store_4d(&tm_o, s_o + x * (kBM * 128), x * 64, row0, h, b);
      tma_store_commit();
      tma_store_wait_all();
    }
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int D, bool kBF16>
static cudaError_t launch_one(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                              const CUtensorMap& o, const PrefillParams& p, int grid,
                              cudaStream_t stream) {
  auto kern = prefill_fwd_kernel<D, kBF16>;
  static bool configured = false;  // per template instance
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  kern<<<grid, kThreads, Cfg<D>::kSmemBytes, stream>>>(q, k, v, o, p);
  return cudaGetLastError();
}

cudaError_t prefill_launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const CUtensorMap& o, const PrefillParams& p, int D, bool bf16,
                           cudaStream_t stream) {
  const int grid = p.B * p.H * p.num_q_blocks;
  if (grid == 0) return cudaSuccess;
  if (D == 128) return bf16 ? launch_one<128, true>(q, k, v, o, p, grid, stream)
                            : launch_one<128, false>(q, k, v, o, p, grid, stream);
  return bf16 ? launch_one<64, true>(q, k, v, o, p, grid, stream)
              : launch_one<64, false>(q, k, v, o, p, grid, stream);
}

int prefill_rows_per_cta() { return kTiles * kBM; }
int prefill_box_rows() { return kBM; }

}  // namespace attn_sm103a
