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
// A CTA owns a block of query rows, whose E4M3 Q rows stay resident in shared
// memory as kSlabs slabs of 128 (query, head) pairs (R = 128 / H rows each),
// together with their weights and windows, and walks a contiguous range of
// 128-key tiles that a producer warp streams through a 4-stage ring (the
// page's split of the key axis across the grid).  Per (key tile, slab) one
// tcgen05.mma .kind::f8f6f4 chain computes S^T = K_tile Q_slab^T, M = 128 keys
// by N = 128 pairs, into one of four 128-column tensor-memory buffers; three
// epilogue warpgroups take the (tile, slab) units round-robin, so the MMA runs
// ahead while a sub-partition's three epilogue warps hide each other's loads.
//
// Epilogue: each thread owns one key (its tensor-memory lane) and reads all
// 128 of the slab's columns as two 64-column loads, so the weighted head sum
// stays inside the thread, and every weight load is a 16-byte broadcast
// serving 4 columns.  For keys with a non-negative scale the ReLU needs no
// scale at all (it factors out of the head sum) and is split across two
// pipes (an integer max on the ALU for half of the columns, an exact
// saturating multiply on the FMA pipe for the other half; see
// accumulate64); the weighted sum is a packed FMA.  Stores run along the key
// axis (128 contiguous bytes per row and warp).  A (tile, slab) pair none of whose rows' windows meets the tile is
// neither multiplied nor read back (the page's tile_skip / empty-window fix);
// a tile no slab needs is not even loaded.  Every wait is bounded.
#include "mqa_logits_sm103a.h"
#include "host_once.h"
#include "sm103a_ptx.cuh"

#include <climits>

namespace attn_sm103a {

namespace {

constexpr int kD = 128;           // head dimension (bytes per E4M3 row)
constexpr int kKeys = 128;        // keys per tile (MMA M)
constexpr int kCols = 128;        // (query, head) pairs per slab (MMA N)
constexpr int kSlabs = 8;         // resident slabs per query block
constexpr int kKRing = 4;         // key-tile stages
constexpr int kBufs = 4;          // tensor-memory buffers of kCols columns
constexpr int kEpiGroups = 3;     // epilogue warpgroups: unit v goes to v % 3
constexpr int kEpiWarps = 4 * kEpiGroups;
constexpr int kThreads = 32 * kEpiWarps + 128;  // 12 epilogue warps | producer, MMA, 2 idle
constexpr int kWarpLoad = kEpiWarps;
constexpr int kWarpMma = kEpiWarps + 1;
constexpr int kTile = kKeys * kD;  // 16 KB: one key tile or one Q slab
// Registers are granted per warpgroup: the block launches with 128 per thread
// (65536 in all) and setmaxnreg gives the three epilogue warpgroups 152, the
// control warpgroup 56 (3*128*152 + 128*56 = 65536).
constexpr int kRegsLaunch = 128;
constexpr int kRegsEpi = 152;
constexpr int kRegsCtl = 56;
static_assert(kEpiGroups * 128 * kRegsEpi + 128 * kRegsCtl <= kThreads * kRegsLaunch,
              "register split exceeds the block's launch allocation");
static_assert(kCols * kD == kTile, "a slab and a key tile have the same size");
static_assert(kSlabs >= kEpiGroups, "every warpgroup sees every key tile");

struct alignas(16) Stats {
  float w[kSlabs * kCols];             // weights of the block's (query, head) pairs
  int lo[kSlabs * 4], hi[kSlabs * 4];  // clamped windows of the block's rows (R <= 4)
  int slo[kSlabs], shi[kSlabs];        // per slab: [min lo, max hi) of its non-empty windows
};

constexpr int kOffQ = 0;
constexpr int kOffK = kSlabs * kTile;
constexpr int kOffStats = kOffK + kKRing * kTile;
constexpr int kOffCtl = kOffStats + static_cast<int>(sizeof(Stats));

struct Ctl {
  uint64_t q_full;             // Q slabs landed, stats written
  uint64_t k_full[kKRing];
  uint64_t k_empty[kKRing];    // MMA commit after the tile's last slab
  uint64_t s_full[kBufs];      // MMA commit per (tile, slab)
  uint64_t t_empty[kBufs];     // the 4 warps of the unit's warpgroup hold the buffer in registers
  uint64_t mma_done;
  uint64_t tmem_free;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Ctl) <= 256, "control block must fit its reserved bytes");
static_assert(kOffStats % 16 == 0 && kOffCtl % 8 == 0, "stats and barriers stay aligned");
constexpr int kSmem = kOffCtl + 256 + 1024;

// A slab takes part in a key tile when some row's window meets it; empty
// slabs carry slo = INT_MAX, shi = INT_MIN and never do.
__device__ __forceinline__ bool slab_live(int slo, int shi, int key0) {
  return slo < key0 + kKeys && shi > key0;
}

// Fast path (scale >= 0 and finite): relu(scale * x) = scale * relu(x), so
// every element needs only relu(x) and the key's scale multiplies the head
// sum once.  The ReLU is split across two pipes: for half of the columns an
// integer max with 0 on the float's bits (negative floats, -0 included, are
// negative integers; ALU pipe), for the other half a saturating multiply by
// 2^-25 (FMA pipe).  For E4M3 operands |q.k| <= 128 * 448^2 < 2^25, so
// x * 2^-25 lies in (-1, 1): the saturation clamps exactly the negative part
// to 0 and, being a power of two, rounds nothing; that half's head sum is
// scaled back by 2^25.  Keys with a negative or non-finite scale take the
// plain multiply-and-max form.
constexpr float kSatDown = 0x1p-25f;
constexpr float kSatUp = 0x1p25f;

// One 64-column read of a unit: x holds this thread's key at slab columns
// C0 .. C0 + 63.  Weights are the same for every key, so each 16-byte
// shared-memory load is a broadcast serving 4 columns.  ai / as accumulate
// per slab row (column pairs packed, f32x2): the integer-max columns and the
// saturating columns on the fast path, simply the even and odd column pairs
// of each group of 4 otherwise.
template <int H, int C0, bool kFast>
__device__ __forceinline__ void accumulate64(const float (&x)[64], const float* w_slab, float scale,
                                             uint64_t (&ai)[kCols / H], uint64_t (&as)[kCols / H]) {
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int row = (C0 + 4 * k) / H;  // a group of 4 columns never straddles rows (H % 4 == 0)
    const float4 w4 = *reinterpret_cast<const float4*>(w_slab + C0 + 4 * k);
    float y0, y1, y2, y3;
    if (kFast) {
      y0 = __int_as_float(max(__float_as_int(x[4 * k]), 0));
      y1 = __int_as_float(max(__float_as_int(x[4 * k + 1]), 0));
      y2 = mul_sat(x[4 * k + 2], kSatDown);
      y3 = mul_sat(x[4 * k + 3], kSatDown);
    } else {
      y0 = fmaxf(x[4 * k] * scale, 0.f);
      y1 = fmaxf(x[4 * k + 1] * scale, 0.f);
      y2 = fmaxf(x[4 * k + 2] * scale, 0.f);
      y3 = fmaxf(x[4 * k + 3] * scale, 0.f);
    }
    ai[row] = f2_fma(f2_pack(y0, y1), f2_pack(w4.x, w4.y), ai[row]);
    as[row] = f2_fma(f2_pack(y2, y3), f2_pack(w4.z, w4.w), as[row]);
  }
}

// The head sums of one unit for this thread's key: z[r] for the slab's rows.
template <int H, bool kFast>
__device__ __forceinline__ void unit_sums(uint32_t taddr, const float* w_slab, float scale,
                                          uint64_t* t_empty, int lane, float (&z)[kCols / H]) {
  constexpr int R = kCols / H;
  uint64_t ai[R], as[R];
#pragma unroll
  for (int r = 0; r < R; ++r) ai[r] = as[r] = f2_pack(0.f, 0.f);
  float x[64];
  tmem_ld64_wait(taddr, x);
  accumulate64<H, 0, kFast>(x, w_slab, scale, ai, as);
  tmem_ld64_wait(taddr + 64, x);
  // The whole buffer is in registers: hand it back.
  tc_fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive(t_empty);
  accumulate64<H, 64, kFast>(x, w_slab, scale, ai, as);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float i0, i1, s0, s1;
    f2_unpack(ai[r], i0, i1);
    f2_unpack(as[r], s0, s1);
    z[r] = kFast ? scale * fmaf(s0 + s1, kSatUp, i0 + i1) : (i0 + i1) + (s0 + s1);
  }
}

template <int H>
__global__ void __launch_bounds__(kThreads, 1)
    mqa_logits_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const MqaParams p) {
  constexpr int R = kCols / H;         // query rows per slab
  constexpr int kRows = kSlabs * R;    // query rows per block (<= 32)
  static_assert(kRows <= 32 && R <= 4, "a block's rows fit one warp's lanes");
  extern __shared__ uint8_t smem_raw[];
  // Offset from the __shared__ array (not integer arithmetic on its address),
  // so the compiler keeps every access in the shared state space.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Stats* stats = reinterpret_cast<Stats*>(smem + kOffStats);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kOffCtl);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const int row0 = blockIdx.x * kRows;
  const int n_tiles = (p.S_kv + kKeys - 1) / kKeys;
  const int t_begin = blockIdx.y * p.tiles_per_cta;
  const int n_t = max(0, min(p.tiles_per_cta, n_tiles - t_begin));

  if (warp == kWarpMma) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < kKRing; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
    }
    for (int b = 0; b < kBufs; ++b) {
      mbar_init(&ctl->s_full[b], 1);
      mbar_init(&ctl->t_empty[b], 4);
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

  if (warp >= kEpiWarps) {
   setmaxnreg_dec<kRegsCtl>();
   if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    if (n_t > 0) {
      // The block's weights (rows are consecutive in w), windows and per-slab
      // window bounds, then its Q slabs; rows past S_q get weight 0, an empty
      // window and zero-filled Q rows.
#pragma unroll 8
      for (int e = 0; e < kSlabs * kCols / 32; ++e) {
        const int idx = lane + 32 * e;
        stats->w[idx] = row0 + idx / H < p.S_q ? p.w[static_cast<size_t>(row0) * H + idx] : 0.f;
      }
      int lo = 0, hi = 0;
      if (lane < kRows && row0 + lane < p.S_q) {
        lo = max(p.start[row0 + lane], 0);
        hi = min(p.end[row0 + lane], p.S_kv);
      }
      if (lo >= hi) lo = hi = 0;
      int blo = lo < hi ? lo : INT_MAX, bhi = lo < hi ? hi : INT_MIN;
#pragma unroll
      for (int o = 1; o < R; o <<= 1) {
        blo = min(blo, __shfl_xor_sync(0xffffffffu, blo, o));
        bhi = max(bhi, __shfl_xor_sync(0xffffffffu, bhi, o));
      }
      if (lane < kRows) {
        stats->lo[lane] = lo;
        stats->hi[lane] = hi;
        if (lane % R == 0) {
          stats->slo[lane / R] = blo;
          stats->shi[lane / R] = bhi;
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&ctl->q_full, kSlabs * kTile);
        for (int s = 0; s < kSlabs; ++s)
          tma_load_2d(smem + kOffQ + s * kTile, &tm_q, &ctl->q_full, 0, (row0 + s * R) * H);
      }
      const int my_slo = lane < kSlabs ? stats->slo[lane] : INT_MAX;
      const int my_shi = lane < kSlabs ? stats->shi[lane] : INT_MIN;
      int issued = 0;
      for (int tl = 0; tl < n_t; ++tl) {
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        const int stg = tl % kKRing;
        const int key0 = (t_begin + tl) * kKeys;
        const bool live = __any_sync(0xffffffffu, slab_live(my_slo, my_shi, key0));
        bool ok = true;
        if (lane == 0 && tl >= kKRing)
          ok = mbar_wait(&ctl->k_empty[stg], (tl / kKRing - 1) & 1, p.wait_limit_ns, p.err, 150);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&ctl->k_full[stg], live ? kTile : 0);
          if (live) tma_load_2d(smem + kOffK + stg * kTile, &tm_k, &ctl->k_full[stg], 0, key0);
        }
        issued = tl + 1;
      }
      if (lane == 0) {  // no copy may still be landing when the CTA exits
        for (int tl = max(0, issued - kKRing); tl < issued; ++tl)
          mbar_wait(&ctl->k_full[tl % kKRing], (tl / kKRing) & 1, p.wait_limit_ns, p.err, 151);
        mbar_wait(&ctl->q_full, 0, p.wait_limit_ns, p.err, 152);
      }
    }
    __syncwarp();
   } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_t > 0) {
      constexpr uint32_t idesc = idesc_e4m3(kKeys, kCols, false, false);
      const uint32_t hi = sdesc_hi_sw128(1024);
      const uint32_t q_lo0 = sdesc_lo(smem_u32(smem + kOffQ), 16);
      const uint32_t k_lo0 = sdesc_lo(smem_u32(smem + kOffK), 16);
      bool ok = mbar_wait(&ctl->q_full, 0, p.wait_limit_ns, p.err, 160);
      for (int tl = 0; tl < n_t && ok; ++tl) {
        const int stg = tl % kKRing;
        const int key0 = (t_begin + tl) * kKeys;
        if (!(ok = mbar_wait(&ctl->k_full[stg], (tl / kKRing) & 1, p.wait_limit_ns, p.err, 161)))
          break;
        const uint32_t k_lo = k_lo0 + ((stg * kTile) >> 4);
#pragma unroll
        for (int s = 0; s < kSlabs; ++s) {
          const int v = tl * kSlabs + s, b = v % kBufs;
          if (v >= kBufs && !(ok = mbar_wait(&ctl->t_empty[b], (v / kBufs - 1) & 1,
                                             p.wait_limit_ns, p.err, 162)))
            break;
          tc_fence_after_sync();
          if (slab_live(stats->slo[s], stats->shi[s], key0)) {
            const uint32_t q_lo = q_lo0 + ((s * kTile) >> 4);
#pragma unroll
            for (int kk = 0; kk < kD / 32; ++kk)
              mma_ss_lh<true>(tmem + kCols * b, k_lo + ((kk * 32) >> 4), hi,
                              q_lo + ((kk * 32) >> 4), hi, idesc, kk > 0);
          }
          mma_commit(&ctl->s_full[b]);
        }
        if (!ok) break;
        mma_commit(&ctl->k_empty[stg]);
      }
      if (!ok) *abort_flag = 1;
      mma_commit(&ctl->mma_done);
      mbar_wait(&ctl->mma_done, 0, p.wait_limit_ns, p.err, 163);
    }
    __syncwarp();
    mbar_wait(&ctl->tmem_free, 0, p.wait_limit_ns, p.err, 164);
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
   }
  } else {
    setmaxnreg_inc<kRegsEpi>();
    // ------------------------------------------------------------ epilogue
    const int wg = warp / 4;       // this warpgroup's units: wg, wg + 3, ...
    const int quad = warp % 4;     // tensor-memory lanes 32 quad .. 32 quad + 31
    const int jl = quad * 32 + lane;  // this thread's key within a tile
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    bool ok = true;
    if (n_t > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->q_full, 0, p.wait_limit_ns, p.err, 173));
    // The next tile's scale of this thread's key is loaded a tile ahead, so
    // the load's latency stays hidden.
    float next_scale = 0.f;
    auto fetch_scale = [&](int tl) {
      const int j = (t_begin + tl) * kKeys + jl;
      next_scale = j < p.S_kv ? p.kv_scale[j] : 0.f;
    };
    if (n_t > 0) fetch_scale(0);
    // This warpgroup's units in order: v = wg, wg + 3, ... (tile v / kSlabs,
    // slab v % kSlabs, buffer v % kBufs).  A unit is read as two 64-column
    // halves; the latency of each load is covered by the other epilogue warps
    // of the SM sub-partition.
    const int n_units = n_t * kSlabs;
    float scale = 0.f;
    bool fast = true;
    int cur_tl = -1;
    for (int v = wg; v < n_units && ok; v += kEpiGroups) {
      const int tl = v / kSlabs, s = v % kSlabs, b = v % kBufs;
      const int key0 = (t_begin + tl) * kKeys;
      if (tl != cur_tl) {  // this warpgroup visits every tile, in order
        cur_tl = tl;
        scale = next_scale;
        if (tl + 1 < n_t) fetch_scale(tl + 1);
        // The path is chosen per warp, never per thread: it holds
        // warp-collective tensor-memory loads (.sync.aligned), __syncwarp and
        // the barrier arrive, which the whole warp must reach together.
        fast = __all_sync(0xffffffffu, scale >= 0.f && scale <= 3.0e38f);
      }
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&ctl->s_full[b], (v / kBufs) & 1, p.wait_limit_ns, p.err, 170));
      if (!ok) break;
      tc_fence_after_sync();
      float z[R];
      const float* w_slab = stats->w + s * kCols;
      const uint32_t taddr = lane_addr + kCols * b;
      if (slab_live(stats->slo[s], stats->shi[s], key0)) {
        if (fast)
          unit_sums<H, true>(taddr, w_slab, scale, &ctl->t_empty[b], lane, z);
        else
          unit_sums<H, false>(taddr, w_slab, scale, &ctl->t_empty[b], lane, z);
      } else {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->t_empty[b]);
#pragma unroll
        for (int r = 0; r < R; ++r) z[r] = 0.f;
      }
      // Each row's 32 keys of this warp are 128 contiguous bytes.
      const int j = key0 + jl;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int lr = s * R + r;
        const int i = row0 + lr;
        const bool inside = j >= stats->lo[lr] && j < stats->hi[lr];
        if (i < p.S_q && j < p.S_kv && (inside || p.clean))
          p.logits[static_cast<size_t>(i) * p.stride + j] = inside ? z[r] : -INFINITY;
      }
    }
    if (ok && n_t > 0)
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
  static std::atomic<unsigned long long> configured{0};  // per template instance, per device
  cudaError_t ce = attn_host::once_per_device(configured, [&]() {
    // The in-kernel register split assumes exactly kRegsLaunch registers per
    // thread at launch; with fewer, setmaxnreg.inc would never complete.
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (ce != cudaSuccess) return ce;
  kern<<<grid, kThreads, kSmem, stream>>>(q, k, p);
  return cudaGetLastError();
}

}  // namespace

int mqa_rows_per_block(int H) { return kSlabs * (kCols / H); }
int mqa_keys_per_tile() { return kKeys; }
int mqa_rows_per_slab_box() { return kCols; }

int mqa_tiles_per_cta(int S_q, int S_kv, int H, int num_sms) {
  // Split the key axis so that the grid fills whole waves of one CTA per SM:
  // minimise waves x (tiles per CTA + the fixed cost of a CTA, about three
  // tiles' worth of loading Q and setting up).
  const int64_t blocks = (S_q + mqa_rows_per_block(H) - 1) / mqa_rows_per_block(H);
  const int64_t tiles = (S_kv + kKeys - 1) / kKeys;
  if (blocks == 0 || tiles == 0) return 1;
  int64_t best_tpc = tiles, best_cost = INT64_MAX;
  // Beyond ~16 waves more splits only add per-CTA cost.
  int64_t max_splits = (16 * static_cast<int64_t>(num_sms) + blocks - 1) / blocks;
  if (max_splits > tiles) max_splits = tiles;
  if (max_splits > 65535) max_splits = 65535;
  for (int64_t splits = 1; splits <= max_splits; ++splits) {
    const int64_t tpc = (tiles + splits - 1) / splits;
    if (splits > 1 && (tiles + tpc - 1) / tpc != splits) continue;  // same grid as a smaller split
    const int64_t waves = (blocks * splits + num_sms - 1) / num_sms;
    const int64_t cost = waves * (tpc + 3);
    if (cost < best_cost) {
      best_cost = cost;
      best_tpc = tpc;
    }
  }
  return static_cast<int>(best_tpc);
}

cudaError_t mqa_logits_launch(const CUtensorMap& q, const CUtensorMap& k, const MqaParams& p,
                              cudaStream_t stream) {
  const int rows = mqa_rows_per_block(p.H);
  const int tiles = (p.S_kv + kKeys - 1) / kKeys;
  if (p.tiles_per_cta <= 0) return cudaErrorInvalidValue;
  const dim3 grid((p.S_q + rows - 1) / rows, (tiles + p.tiles_per_cta - 1) / p.tiles_per_cta);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  switch (p.H) {
    case 32: return launch_h<32>(q, k, p, grid, stream);
    case 64: return launch_h<64>(q, k, p, grid, stream);
    case 128: return launch_h<128>(q, k, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn_sm103a
