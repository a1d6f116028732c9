// mqa_logits_sm103a.cu -- FP8 MQA logits for sm_103a, D = 128.
//
//   logits[i,j] = sum_h w[i,h] * max(0, kv_scale[j] * (q[i,h] . k[j]))
//
// for j in row i's key window [start_i, end_i) (clamped to [0, S_kv)); -inf
// outside it when clean_logits is set, untouched otherwise ("[FlyDSL] FP8 MQA
// logits improvements for gfx950", aiter PR 7412: the per-head products, the
// weighted head reduction, per-key scales, the windows and clean_logits; the
// formula itself is a reading of those pieces).
//
// A CTA owns 128 keys (its E4M3 K tile stays in shared memory) and walks a
// chunk of query groups, G = 256 / H query rows each.  Per group one
// tcgen05.mma .kind::f8f6f4 computes S^T = K_tile Q_group^T with M = 128 keys
// and N = G*H = 256 (query, head) pairs into one of two 256-column
// tensor-memory buffers, so one thread owns one key and reduces over heads in
// its own registers while the MMA of the next group runs.  A group whose
// rows' windows all miss the key tile is neither loaded nor multiplied (the
// page's tile_skip / empty-window fix); with clean_logits its entries are
// still filled with -inf.  Eight epilogue warps split each group's query
// rows (a warp's rows own 128 contiguous tensor-memory columns, read with one
// load); their stores run along the key axis, so every warp writes 128
// contiguous bytes per row.  Every wait is bounded.
#include "mqa_logits_sm103a.h"
#include "sm103a_ptx.cuh"

namespace attn_sm103a {

namespace {

constexpr int kD = 128;           // head dimension (bytes per E4M3 row)
constexpr int kKeys = 128;        // keys per CTA (MMA M)
constexpr int kN = 256;           // (query, head) pairs per group (MMA N)
constexpr int kRing = 4;          // query-group stages
constexpr int kThreads = 384;     // 8 epilogue warps | producer, MMA, 2 idle
constexpr int kEpiWarps = 8;
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr int kKTile = kKeys * kD;   // 16 KB
constexpr int kQTile = kN * kD;      // 32 KB

struct alignas(16) Stage {  // 16-byte aligned: the weights are read as float4
  float w[kN];      // weights of the group's (query, head) pairs
  int lo[8], hi[8]; // clamped windows of the group's rows (G <= 8)
  int live;         // some row's window meets this CTA's keys
};

constexpr int kOffQ = kKTile;
constexpr int kOffStage = kOffQ + kRing * kQTile;
constexpr int kOffCtl = kOffStage + kRing * static_cast<int>(sizeof(Stage));

struct Ctl {
  uint64_t k_full;
  uint64_t full[kRing];
  uint64_t empty[kRing];    // MMA commit + every epilogue warp
  uint64_t s_full[2];
  uint64_t t_empty[2];      // the epilogue warps are done with buffer b
  uint64_t mma_done;
  uint64_t tmem_free;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Ctl) <= 256, "control block must fit its reserved bytes");
static_assert(sizeof(Stage) % 16 == 0 && kOffStage % 16 == 0, "stages must stay 16-byte aligned");
constexpr int kSmem = kOffCtl + 256 + 1024;

template <int H>
__global__ void __launch_bounds__(kThreads, 1)
    mqa_logits_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const MqaParams p) {
  constexpr int G = kN / H;  // query rows per group
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Stage* stages = reinterpret_cast<Stage*>(smem + kOffStage);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kOffCtl);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const int key0 = blockIdx.x * kKeys;
  const int n_groups = (p.S_q + G - 1) / G;
  const int g_begin = blockIdx.y * p.groups_per_cta;
  const int n_u = max(0, min(p.groups_per_cta, n_groups - g_begin));

  if (warp == kWarpMma) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&ctl->k_full, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1 + kEpiWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->s_full[b], 1);
      mbar_init(&ctl->t_empty[b], kEpiWarps);
    }
    mbar_init(&ctl->mma_done, 1);
    mbar_init(&ctl->tmem_free, kEpiWarps);
    ctl->abort = 0;
    fence_mbar_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort;

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    if (n_u > 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&ctl->k_full, kKTile);
        tma_load_2d(smem, &tm_k, &ctl->k_full, 0, key0);
      }
      // A group's windows and weights come from global memory; they are
      // loaded one group ahead, before the wait for the ring slot, so their
      // latency hides behind it instead of serializing the producer.
      constexpr int kWPerLane = kN / 32;
      int nlo = 0, nhi = 0;
      float nw[kWPerLane];
      auto fetch = [&](int u) {
        const int i0 = (g_begin + u) * G;
        nlo = nhi = 0;
        if (lane < G && i0 + lane < p.S_q) {
          nlo = p.start[i0 + lane];
          nhi = p.end[i0 + lane];
        }
#pragma unroll
        for (int e = 0; e < kWPerLane; ++e) {
          const int c = lane + 32 * e;
          const int i = i0 + c / H;
          nw[e] = i < p.S_q ? p.w[static_cast<size_t>(i) * H + c % H] : 0.f;
        }
      };
      fetch(0);
      int issued = 0;
      for (int u = 0; u < n_u; ++u) {
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        const int st = u % kRing;
        const int i0 = (g_begin + u) * G;
        int lo = max(nlo, 0), hi = min(nhi, p.S_kv);
        float w[kWPerLane];
#pragma unroll
        for (int e = 0; e < kWPerLane; ++e) w[e] = nw[e];
        if (u + 1 < n_u) fetch(u + 1);
        bool ok = true;
        if (lane == 0 && u >= kRing)
          ok = mbar_wait(&ctl->empty[st], (u / kRing - 1) & 1, p.wait_limit_ns, p.err, 150);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        Stage& sg = stages[st];
        bool live = false;
        if (lane < G) {
          if (i0 + lane >= p.S_q) lo = hi = 0;
          sg.lo[lane] = lo;
          sg.hi[lane] = hi;
          live = lo < hi && lo < key0 + kKeys && hi > key0;
        }
        live = __any_sync(0xffffffffu, live);
#pragma unroll
        for (int e = 0; e < kWPerLane; ++e) sg.w[lane + 32 * e] = w[e];
        if (lane == 0) sg.live = live ? 1 : 0;
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&ctl->full[st], live ? kQTile : 0);
          if (live) tma_load_2d(smem + kOffQ + st * kQTile, &tm_q, &ctl->full[st], 0, i0 * H);
        }
        issued = u + 1;
      }
      if (lane == 0) {  // no copy may still be landing when the CTA exits
        for (int u = max(0, issued - kRing); u < issued; ++u)
          mbar_wait(&ctl->full[u % kRing], (u / kRing) & 1, p.wait_limit_ns, p.err, 151);
        mbar_wait(&ctl->k_full, 0, p.wait_limit_ns, p.err, 152);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_u > 0) {
      constexpr uint32_t idesc = idesc_e4m3(kKeys, kN, false, false);
      const uint32_t hi = sdesc_hi_sw128(1024);
      const uint32_t k_lo = sdesc_lo(smem_u32(smem), 16);
      bool ok = mbar_wait(&ctl->k_full, 0, p.wait_limit_ns, p.err, 160);
      for (int u = 0; u < n_u && ok; ++u) {
        const int st = u % kRing, b = u & 1;
        if (!(ok = mbar_wait(&ctl->full[st], (u / kRing) & 1, p.wait_limit_ns, p.err, 161)))
          break;
        if (u >= 2 &&
            !(ok = mbar_wait(&ctl->t_empty[b], (u / 2 - 1) & 1, p.wait_limit_ns, p.err, 162)))
          break;
        tc_fence_after_sync();
        if (stages[st].live) {
          const uint32_t q_lo = sdesc_lo(smem_u32(smem + kOffQ + st * kQTile), 16);
#pragma unroll
          for (int kk = 0; kk < kD / 32; ++kk)
            mma_ss_lh<true>(tmem + 256 * b, k_lo + ((kk * 32) >> 4), hi,
                            q_lo + ((kk * 32) >> 4), hi, idesc, kk > 0);
        }
        mma_commit(&ctl->s_full[b]);
        mma_commit(&ctl->empty[st]);
      }
      if (!ok) *abort_flag = 1;
      mma_commit(&ctl->mma_done);
      mbar_wait(&ctl->mma_done, 0, p.wait_limit_ns, p.err, 163);
    }
    __syncwarp();
    mbar_wait(&ctl->tmem_free, 0, p.wait_limit_ns, p.err, 164);
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  } else if (warp < kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int half = warp / 4;                 // this warp's half of the group's rows
    const int r = (warp % 4) * 32 + lane;      // key within the tile
    const int j = key0 + r;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    const float scale = j < p.S_kv ? p.kv_scale[j] : 0.f;
    bool ok = true;
    for (int u = 0; u < n_u; ++u) {
      const int st = u % kRing, b = u & 1;
      // The stage's statistics come from the producer (its full barrier), the
      // scores from the MMA warp (s_full).
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&ctl->full[st], (u / kRing) & 1, p.wait_limit_ns, p.err, 172) &&
                          mbar_wait(&ctl->s_full[b], (u / 2) & 1, p.wait_limit_ns, p.err, 170));
      if (!ok) break;
      tc_fence_after_sync();
      const Stage& sg = stages[st];
      const bool live = sg.live != 0;
      const int i0 = (g_begin + u) * G;
      // This warp's rows of the group own 128 contiguous columns of the
      // buffer: one load, one wait.
      float sv[128];
      if (live) tmem_ld128_wait(lane_addr + 256 * b + 128 * half, sv);
      const uint64_t sc2 = f2_pack(scale, scale);
#pragma unroll
      for (int gg = 0; gg < G / 2; ++gg) {
        const int g = half * (G / 2) + gg;
        const int i = i0 + g;
        float acc = 0.f;
        if (live) {
          uint64_t a0 = f2_pack(0.f, 0.f), a1 = a0;
#pragma unroll
          for (int c = 0; c < H; c += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(&sg.w[g * H + c]);
            float x0, x1, x2, x3;
            f2_unpack(f2_mul(f2_pack(sv[gg * H + c], sv[gg * H + c + 1]), sc2), x0, x1);
            f2_unpack(f2_mul(f2_pack(sv[gg * H + c + 2], sv[gg * H + c + 3]), sc2), x2, x3);
            a0 = f2_fma(f2_pack(fmaxf(x0, 0.f), fmaxf(x1, 0.f)), f2_pack(w4.x, w4.y), a0);
            a1 = f2_fma(f2_pack(fmaxf(x2, 0.f), fmaxf(x3, 0.f)), f2_pack(w4.z, w4.w), a1);
          }
          float p0, p1, p2, p3;
          f2_unpack(a0, p0, p1);
          f2_unpack(a1, p2, p3);
          acc = (p0 + p1) + (p2 + p3);
        }
        if (i < p.S_q && j < p.S_kv) {
          const bool inside = j >= sg.lo[g] && j < sg.hi[g];
          float* dst = p.logits + static_cast<size_t>(i) * p.stride + j;
          if (inside)
            *dst = acc;
          else if (p.clean)
            *dst = -INFINITY;
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl->t_empty[b]);
        mbar_arrive(&ctl->empty[st]);
      }
    }
    if (ok && n_u > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->mma_done, 0, p.wait_limit_ns, p.err, 171));
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->tmem_free);
  }
}

template <int H>
cudaError_t launch_h(const CUtensorMap& q, const CUtensorMap& k, const MqaParams& p, dim3 grid,
                     cudaStream_t stream) {
  auto kern = mqa_logits_kernel<H>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  kern<<<grid, kThreads, kSmem, stream>>>(q, k, p);
  return cudaGetLastError();
}

}  // namespace

int mqa_rows_per_group(int H) { return kN / H; }
int mqa_keys_per_cta() { return kKeys; }

cudaError_t mqa_logits_launch(const CUtensorMap& q, const CUtensorMap& k, const MqaParams& p,
                              cudaStream_t stream) {
  const int G = kN / p.H;
  const int n_groups = (p.S_q + G - 1) / G;
  const dim3 grid((p.S_kv + kKeys - 1) / kKeys, (n_groups + p.groups_per_cta - 1) / p.groups_per_cta);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  switch (p.H) {
    case 32: return launch_h<32>(q, k, p, grid, stream);
    case 64: return launch_h<64>(q, k, p, grid, stream);
    case 128: return launch_h<128>(q, k, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn_sm103a
