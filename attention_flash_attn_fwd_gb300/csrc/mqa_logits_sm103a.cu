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
// Epilogue: each warp reads its 32 keys of a buffer as two 16x256b loads, so
// a thread holds 4 keys x 32 of the slab's 128 columns and every weight it
// reads from shared memory serves 4 keys.  The ReLU is split across two pipes
// (an integer max on the ALU for one key of a register pair, an exact
// saturating multiply on the FMA pipe for the other; see KeyScale), the
// weighted sum is a packed FMA, and two shuffle steps finish the head sum
// across the 4 threads that share a key.  Stores run along the key axis (128 contiguous bytes per row and
// warp).  A (tile, slab) pair none of whose rows' windows meets the tile is
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

// ReLU by saturation.  For E4M3 operands |q.k| <= 128 * 448^2 < 2^25, so with
// |scale| <= 2^e the product x * scale * 2^-(25+e) lies in [-1, 1] and a
// saturating multiply clamps exactly its negative part to 0.  Power-of-two
// scalings round nothing, so sat(x * s_sat) * 2^(25+e) is the rounded
// relu(scale * x) itself, with no max instruction per element.  Scales beyond
// 2^100 (or NaN) fall back to the plain multiply-and-max form.
struct KeyScale {
  float s_sat;    // multiplier applied to every product
  float unscale;  // multiplier applied to the head sum
  bool by_sat;    // the saturating form is exact for this key
};

__device__ __forceinline__ KeyScale key_scale(float scale) {
  KeyScale k;
  int e = 0;
  frexpf(scale, &e);
  e = max(e, -100);
  k.by_sat = fabsf(scale) <= 0x1p100f;
  k.s_sat = k.by_sat ? ldexpf(scale, -(25 + e)) : scale;
  k.unscale = k.by_sat ? ldexpf(1.f, 25 + e) : 1.f;
  return k;
}

// The fast path splits the ReLU between two pipes.  Key g (scale >= 0):
// relu(scale * x) = scale * relu(x), and relu of a float is a signed-integer
// max with 0 on its bits (negative floats, -0 included, are negative
// integers) on the ALU pipe; its head sum is scaled once.  Key g + 8: the
// exact saturating multiply on the FMA pipe (see KeyScale).  Both feed a
// packed f32x2 FMA over the column pairs the load already delivers adjacent.
template <int H>
__device__ __forceinline__ void accumulate_half_pos(const float (&v)[64], const float* w_slab, int c,
                                                    float s_sat1, uint64_t (&a)[kCols / H][2]) {
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int row = (8 * r) / H;
    const float2 w2 = *reinterpret_cast<const float2*>(&w_slab[8 * r + 2 * c]);
    const uint64_t wp = f2_pack(w2.x, w2.y);
    const float y0 = __int_as_float(max(__float_as_int(v[4 * r]), 0));
    const float y1 = __int_as_float(max(__float_as_int(v[4 * r + 1]), 0));
    const float y2 = mul_sat(v[4 * r + 2], s_sat1);
    const float y3 = mul_sat(v[4 * r + 3], s_sat1);
    a[row][0] = f2_fma(f2_pack(y0, y1), wp, a[row][0]);
    a[row][1] = f2_fma(f2_pack(y2, y3), wp, a[row][1]);
  }
}

// One 16-lane half of a warp's 32 keys: v holds keys g (v[4r], v[4r+1]) and
// g + 8 (v[4r+2], v[4r+3]) at slab columns 8r + 2c and 8r + 2c + 1.
// Accumulates w * relu(scale * x) per (row of the slab, key, column parity)
// in scalar registers: one saturating multiply and one FMA per element.
template <int H, bool kSat>
__device__ __forceinline__ void accumulate_half(const float (&v)[64], const float* w_slab, int c,
                                                const KeyScale& k0, const KeyScale& k1,
                                                float (&a)[kCols / H][2][2]) {
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int row = (8 * r) / H;  // a repetition's 8 columns never straddle rows (H % 8 == 0)
    const float2 w2 = *reinterpret_cast<const float2*>(&w_slab[8 * r + 2 * c]);
    float y0, y1, y2, y3;
    if (kSat) {
      y0 = mul_sat(v[4 * r], k0.s_sat);
      y1 = mul_sat(v[4 * r + 1], k0.s_sat);
      y2 = mul_sat(v[4 * r + 2], k1.s_sat);
      y3 = mul_sat(v[4 * r + 3], k1.s_sat);
    } else {
      y0 = fmaxf(v[4 * r] * k0.s_sat, 0.f);
      y1 = fmaxf(v[4 * r + 1] * k0.s_sat, 0.f);
      y2 = fmaxf(v[4 * r + 2] * k1.s_sat, 0.f);
      y3 = fmaxf(v[4 * r + 3] * k1.s_sat, 0.f);
    }
    a[row][0][0] = fmaf(y0, w2.x, a[row][0][0]);
    a[row][0][1] = fmaf(y1, w2.y, a[row][0][1]);
    a[row][1][0] = fmaf(y2, w2.x, a[row][1][0]);
    a[row][1][1] = fmaf(y3, w2.y, a[row][1][1]);
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
    const int g = lane / 4, c = lane % 4;
    // Before the head sum, a thread's keys are (half hf, kp): quad*32 + 16 hf
    // + g + 8 kp; after it, the thread owns one key per row.
    const int j_off = quad * 32 + 16 * (c >> 1) + g + 8 * (c & 1);
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    bool ok = true;
    if (n_t > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->q_full, 0, p.wait_limit_ns, p.err, 173));
    // The next tile's per-key scales are loaded a tile ahead and only turned
    // into KeyScale when that tile starts, so the load's latency stays hidden.
    float nraw[2][2];
    auto fetch_scales = [&](int tl) {
      const int key0 = (t_begin + tl) * kKeys;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int kp = 0; kp < 2; ++kp) {
          const int jj = key0 + quad * 32 + 16 * hf + g + 8 * kp;
          nraw[hf][kp] = jj < p.S_kv ? p.kv_scale[jj] : 0.f;
        }
    };
    if (n_t > 0) fetch_scales(0);
    // This warpgroup's units in order: v = wg, wg + 3, ... (tile v / kSlabs,
    // slab v % kSlabs, buffer v % kBufs).  A unit is read as two 64-register
    // halves; the latency of each load is covered by the other epilogue warps
    // of the SM sub-partition.
    const int n_units = n_t * kSlabs;
    KeyScale ks[2][2];
    float kraw[2][2];
    bool sat = true, pos = true, fast = true;
    int cur_tl = -1;
    for (int v = wg; v < n_units && ok; v += kEpiGroups) {
      const int tl = v / kSlabs, s = v % kSlabs, b = v % kBufs;
      const int key0 = (t_begin + tl) * kKeys;
      if (tl != cur_tl) {  // this warpgroup visits every tile, in order
        cur_tl = tl;
        pos = true;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int kp = 0; kp < 2; ++kp) {
            kraw[hf][kp] = nraw[hf][kp];
            ks[hf][kp] = key_scale(nraw[hf][kp]);
            pos = pos && nraw[hf][kp] >= 0.f && nraw[hf][kp] <= 3.0e38f;
          }
        if (tl + 1 < n_t) fetch_scales(tl + 1);
        sat = ks[0][0].by_sat && ks[0][1].by_sat && ks[1][0].by_sat && ks[1][1].by_sat;
        // The path is chosen per warp, never per thread: the branches hold
        // warp-collective tensor-memory loads (.sync.aligned), __syncwarp and
        // the barrier arrive, which the whole warp must reach together.
        pos = __all_sync(0xffffffffu, pos);
        sat = __all_sync(0xffffffffu, sat);
        fast = pos && sat;
      }
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&ctl->s_full[b], (v / kBufs) & 1, p.wait_limit_ns, p.err, 170));
      if (!ok) break;
      tc_fence_after_sync();
      const bool live = slab_live(stats->slo[s], stats->shi[s], key0);
      float u[2][R][2];  // [half][row][key of the pair]: this thread's partial head sums
      const float* w_slab = stats->w + s * kCols;
      const uint32_t taddr = lane_addr + kCols * b;
      if (live && fast) {
        uint64_t a2[2][R][2];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int r = 0; r < R; ++r) a2[hf][r][0] = a2[hf][r][1] = f2_pack(0.f, 0.f);
        float x[64];
        tmem_ld16x256b_x16_wait(taddr, x);
        accumulate_half_pos<H>(x, w_slab, c, ks[0][1].s_sat, a2[0]);
        tmem_ld16x256b_x16_wait(taddr + (16u << 16), x);
        // The whole buffer is in registers: hand it back.
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->t_empty[b]);
        accumulate_half_pos<H>(x, w_slab, c, ks[1][1].s_sat, a2[1]);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int kp = 0; kp < 2; ++kp) {
              float lo, hi;
              f2_unpack(a2[hf][r][kp], lo, hi);
              u[hf][r][kp] = lo + hi;
            }
      } else if (live) {
        float a[2][R][2][2];  // [half][row][key of the pair][column parity]
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int r = 0; r < R; ++r)
            a[hf][r][0][0] = a[hf][r][0][1] = a[hf][r][1][0] = a[hf][r][1][1] = 0.f;
        float x[64];
        tmem_ld16x256b_x16_wait(taddr, x);
        if (sat)
          accumulate_half<H, true>(x, w_slab, c, ks[0][0], ks[0][1], a[0]);
        else
          accumulate_half<H, false>(x, w_slab, c, ks[0][0], ks[0][1], a[0]);
        tmem_ld16x256b_x16_wait(taddr + (16u << 16), x);
        // The whole buffer is in registers: hand it back.
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->t_empty[b]);
        if (sat)
          accumulate_half<H, true>(x, w_slab, c, ks[1][0], ks[1][1], a[1]);
        else
          accumulate_half<H, false>(x, w_slab, c, ks[1][0], ks[1][1], a[1]);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int kp = 0; kp < 2; ++kp) u[hf][r][kp] = a[hf][r][kp][0] + a[hf][r][kp][1];
      } else {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->t_empty[b]);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int r = 0; r < R; ++r) u[hf][r][0] = u[hf][r][1] = 0.f;
      }
      // Head sum across the 4 threads sharing a key: first over the key pair
      // (lane bit 0 keeps kp = c & 1), then over the halves (bit 1 keeps
      // hf = c >> 1); each step sends the half this thread does not keep.
      float z[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float y[2];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const float u0 = u[hf][r][0], u1 = u[hf][r][1];
          const float keep = (c & 1) ? u1 : u0, send = (c & 1) ? u0 : u1;
          y[hf] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
        }
        const float keep = (c & 2) ? y[1] : y[0], send = (c & 2) ? y[0] : y[1];
        z[r] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
      }
      const float unscale =
          fast ? ((c & 2) ? ((c & 1) ? ks[1][1].unscale : kraw[1][0])
                          : ((c & 1) ? ks[0][1].unscale : kraw[0][0]))
              : ((c & 2) ? ((c & 1) ? ks[1][1].unscale : ks[1][0].unscale)
                         : ((c & 1) ? ks[0][1].unscale : ks[0][0].unscale));
      const int j = key0 + j_off;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int lr = s * R + r;
        const int i = row0 + lr;
        const bool inside = j >= stats->lo[lr] && j < stats->hi[lr];
        if (i < p.S_q && j < p.S_kv && (inside || p.clean))
          p.logits[static_cast<size_t>(i) * p.stride + j] = inside ? z[r] * unscale : -INFINITY;
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
