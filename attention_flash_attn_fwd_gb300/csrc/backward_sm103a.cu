// backward_sm103a.cu -- attention backward (dQ, dK, dV) for sm_103a, D = 128.
//
// The gradients of O = softmax(scale Q K^T + causal mask) V for an upstream
// gradient dO ("Backward Flash Attention", Wave February 2025 Release,
// EvoFormer list; "Functionality & Performance on backward attention",
// Milestones).  With P recomputed from the forward's lse,
//
//     D_i   = dO_i . O_i                      (delta kernel)
//     dS_ij = P_ij (dO_i . v_j - D_i)
//     dV_j  = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i   (dK/dV kernel)
//     dQ_i  = scale sum_j dS_ij k_j                            (dQ kernel)
//
// Two tensor-core kernels, each with one 128-row tile per CTA:
//  * dK/dV: a CTA owns 128 keys (K, V resident in shared memory) and walks the
//    query tiles that see them.  Per tile: S^T = K Q^T and dP^T = V dO^T into
//    tensor memory, signalled apart; one thread per key row turns S^T into P^T
//    first and dP^T into dS^T after (16-bit pairs over each element-wise
//    group's own columns); dV += P^T dO and dK += dS^T Q read P^T / dS^T
//    straight from tensor memory, and the next step's S^T follows dV, so dK
//    and the next dP^T run while the next P^T is computed.  Tensor memory:
//    S^T [0,128), dP^T [128,256), dV [256,384), dK [384,512).
//  * dQ: a CTA owns 128 queries (Q, dO resident) and walks the key tiles they
//    see: S = Q K^T, dP = dO V^T, dS, dQ += dS K.  Tensor memory: S [0,128),
//    dP [128,256), dQ [256,384), dS [384,448).  Pipelined: once the
//    element-wise warps hold a step's S and dP in registers, the next step's
//    products overwrite them while dS is computed; K and V stream through
//    rings of their own (3 and 2 stages); one thread issues S and dP, another
//    dQ += dS K.
// The dQ pass recomputes S and dP (7 MMAs per tile pair instead of 5) so that
// no tile's gradient needs atomic accumulation: results are deterministic.
// A TMA warp streams the walking tiles (dK/dV: a 2-stage ring of (Q, dO)
// pairs), MMA-issuing threads in warps 9 (and 10) issue tcgen05.mma, eight
// warps do the element-wise work (two warpgroups, each taking 64 of the 128
// columns of every row); every wait is bounded in time.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "backward_sm103a.h"
#include "host_once.h"
#include "sm103a_ptx.cuh"

namespace attn_sm103a {

namespace {

constexpr int kT = 128;                    // rows per tile (queries or keys), and D
constexpr int kTile = kT * kT * 2;         // one 16-bit 128 x 128 tile (two 64-column panels)
constexpr int kPanel = kT * 128;           // one 64-column panel: 128 rows x 128 bytes
constexpr int kThreadsB = 384;  // 8 element-wise warps | TMA warp, MMA warp, 2 idle warps
constexpr int kEwWarps = 8;
constexpr int kWarpLoad = 8;
constexpr int kWarpMmaB = 9;
constexpr int kWarpMmaDq = 10;  // dQ kernel: issues dQ += dS K beside warp 9's S and dP
// Registers are granted per warpgroup: the block launches with 168 per
// thread (64512 in all) and setmaxnreg gives the two element-wise warpgroups
// 200, the control warpgroup 104 (2*128*200 + 128*104 = 64512): with less,
// the MMA warp's unrolled issue loops spill.
constexpr int kRegsLaunchB = 168;
constexpr int kRegsEw = 200;
constexpr int kRegsCtl = 104;
static_assert(2 * 128 * kRegsEw + 128 * kRegsCtl <= kThreadsB * kRegsLaunchB,
              "register split exceeds the block's launch allocation");
constexpr int kRing = 2;                   // stages of the walking pair of tiles
constexpr float kLog2e = 1.4426950408889634f;

struct BwdCtl {
  uint64_t res_full;          // the resident pair of tiles has landed
  uint64_t full[kRing];       // walking pair (+ its lse/delta rows) has landed
  uint64_t empty[kRing];      // the MMAs reading a stage are done
  uint64_t s_full;            // dK/dV kernel: S^T of a step is in tensor memory
  uint64_t dp_full;           // dK/dV kernel: dP^T of a step is in tensor memory
  uint64_t p_ready;           // dK/dV kernel: P^T of a step is in tensor memory
  uint64_t ew_done;           // the element-wise pass of a step is in tensor memory
  uint64_t mma_done;          // every MMA of the CTA has completed
  uint64_t tmem_free;         // the element-wise warps are done with tensor memory
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(BwdCtl) <= 256, "control block must fit its reserved bytes");

// Shared memory: resident A (32 KB) | resident B (32 KB) | ring of kRing x
// (two 32 KB tiles) | per stage 2 x 128 floats (lse*log2e, delta) | control.
constexpr int kOffRing = 2 * kTile;
constexpr int kOffRows = kOffRing + kRing * 2 * kTile;
constexpr int kOffCtl = kOffRows + kRing * 2 * kT * 4;
constexpr int kSmemB = kOffCtl + 256 + 1024;

__device__ __forceinline__ void load_tile(void* dst, const CUtensorMap* map, uint64_t* bar,
                                          int row, int h, int b, int bshd) {
  for (int x = 0; x < 2; ++x) {
    void* d = static_cast<uint8_t*>(dst) + x * kPanel;
    if (bshd)
      tma_load_4d(d, map, bar, x * 64, h, row, b);
    else
      tma_load_4d(d, map, bar, x * 64, row, h, b);
  }
}

__device__ __forceinline__ void store_tile(const CUtensorMap* map, const void* src, int row,
                                           int h, int b, int bshd) {
  for (int x = 0; x < 2; ++x) {
    const void* s = static_cast<const uint8_t*>(src) + x * kPanel;
    if (bshd)
      tma_store_4d(map, s, x * 64, h, row, b);
    else
      tma_store_4d(map, s, x * 64, row, h, b);
  }
}

// A . B^T over D = 128 into tensor memory: both operands K-major (128-byte
// swizzle, 8-row groups 1024 B apart), M = N = 128, K = 16 per instruction.
__device__ __forceinline__ void mma_abt(uint32_t d, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                        uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk) {
    const uint32_t off = ((kk / 4) * kPanel + (kk % 4) * 32) >> 4;
    mma_ss_lh(d, a_lo + off, hi, b_lo + off, hi, idesc, kk > 0);
  }
}

// D (+)= A . B with A = 128 x 128 16-bit pairs in tensor memory (columns
// [a, a + 64)) and B = a 128-row tile read MN-major (rows are the K index).
__device__ __forceinline__ void mma_tmem_a(uint32_t d, uint32_t a, uint32_t b_lo, uint32_t hi,
                                           uint32_t idesc, bool acc) {
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk)
    mma_ts_lh(d, a + kk * 8, b_lo + ((kk * 16 * 128) >> 4), hi, idesc,
              (acc || kk > 0) ? 1u : 0u);
}

// Same, with A's two 64-key halves in columns [a, a + 32) and [a + 64, a + 96)
// (each element-wise group's packed pairs over its own fp32 columns).
__device__ __forceinline__ void mma_tmem_a_split(uint32_t d, uint32_t a, uint32_t b_lo,
                                                 uint32_t hi, uint32_t idesc, bool acc) {
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk)
    mma_ts_lh(d, a + kk * 8 + (kk >= 4 ? 32 : 0), b_lo + ((kk * 16 * 128) >> 4), hi, idesc,
              (acc || kk > 0) ? 1u : 0u);
}

// Row-major 16-bit O/dO row r of 128 columns into 128-byte-swizzled staging
// (two 64-column panels), from 64 fp32 values per call (columns [64h, 64h+64)).
template <bool kBF16>
__device__ __forceinline__ void stage_row(uint8_t* tile, int r, int h, const uint32_t (&v)[64],
                                          float mul) {
  uint8_t* sub = tile + h * kPanel + r * 128;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint4 w;
    uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      wp[e] = pack2<kBF16>(__uint_as_float(v[q * 8 + 2 * e]) * mul,
                           __uint_as_float(v[q * 8 + 2 * e + 1]) * mul);
    *reinterpret_cast<uint4*>(sub + ((q ^ (r & 7)) * 16)) = w;
  }
}

// The dK/dV kernel's element-wise pass over one 128 x 128 step, in place in
// tensor memory.  The calling warp owns column group g (columns [64g, 64g +
// 64)) of its 32 rows: S^T (fp32, columns [cs, cs + 128)) -> P^T (16-bit pairs,
// [cs + 64g, cs + 64g + 32)), dP^T (fp32, [cd, cd + 128)) -> dS^T = P^T (dP^T -
// delta) (16-bit pairs, [cd + 64g, cd + 64g + 32)): each group's pairs land on
// its own fp32 columns, already in its registers, so no warp waits for
// another before storing (the MMAs read A from the two 32-column ranges).
// S^T and dP^T arrive separately (`s_full`, `dp_full`): P^T is computed from
// S^T alone, stored and announced on `p_ready`, and only then is dP^T waited
// for and read, so the MMA warp can run dK of the previous step and dP^T of
// this one while P^T is computed.  `lse2_of(c)` / `delta_of(c)` give the row
// statistics of the column pair (c, c + 1) as a float2 (per query column);
// `visible(c)` masks causal and ragged positions and is only evaluated when
// kMasked.  Returns false if the wait for dP^T timed out.
template <bool kBF16, bool kMasked, class Lse, class Delta, class Vis>
__device__ __forceinline__ bool elementwise_step_p_first(uint32_t lane_addr, int g, uint32_t cs,
                                                         uint32_t cd, float c, Lse lse2_of,
                                                         Delta delta_of, Vis visible,
                                                         uint64_t* p_ready, uint64_t* dp_full,
                                                         uint32_t dp_parity, uint64_t limit_ns,
                                                         int* err, int lane) {
  uint32_t x[64], y[64];
  tmem_ld64_wait(lane_addr + cs + 64 * g, x);
  // Column pairs in packed fp32 (f32x2): one instruction per two elements.
  const uint64_t c2 = f2_pack(c, c);
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    uint32_t pp[16];
#pragma unroll
    for (int q = 16 * hf; q < 16 * hf + 16; ++q) {
      const int col0 = 64 * g + 2 * q;
      const float2 l2 = lse2_of(col0);
      float a0, a1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(x[2 * q]), __uint_as_float(x[2 * q + 1])), c2,
                       f2_pack(-l2.x, -l2.y)),
                a0, a1);
      float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
      if constexpr (kMasked) {
        p0 = visible(col0) ? p0 : 0.f;
        p1 = visible(col0 + 1) ? p1 : 0.f;
      }
      x[2 * q] = __float_as_uint(p0);  // P in fp32 for the dS phase
      x[2 * q + 1] = __float_as_uint(p1);
      pp[q - 16 * hf] = pack2<kBF16>(p0, p1);
    }
    tmem_st16(lane_addr + cs + 64 * g + 16 * hf, pp);
  }
  tmem_st_wait();
  tc_fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive(p_ready);
  if (!__all_sync(0xffffffffu, mbar_wait(dp_full, dp_parity, limit_ns, err, 72))) return false;
  tc_fence_after_sync();
  tmem_ld64_wait(lane_addr + cd + 64 * g, y);
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    uint32_t dd[16];
#pragma unroll
    for (int q = 16 * hf; q < 16 * hf + 16; ++q) {
      const float2 dl = delta_of(64 * g + 2 * q);
      // dS = P (dP - delta), as (dP - delta) then P * that, both packed
      const uint64_t t = f2_add(f2_pack(__uint_as_float(y[2 * q]), __uint_as_float(y[2 * q + 1])),
                                f2_pack(-dl.x, -dl.y));
      float d0, d1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(x[2 * q]), __uint_as_float(x[2 * q + 1])), t,
                       f2_pack(0.f, 0.f)),
                d0, d1);
      dd[q - 16 * hf] = pack2<kBF16>(d0, d1);
    }
    tmem_st16(lane_addr + cd + 64 * g + 16 * hf, dd);
  }
  tmem_st_wait();
  return true;
}

// ---------------------------------------------------------------- delta

// delta[b,h,i] = sum_d dO[b,h,i,d] * O[b,h,i,d] in fp32.  HBM-bound: 16
// lanes read a row as 16-byte pieces (o and dout are 16-byte aligned,
// checked on the host), a warp takes kDeltaRows rows and issues all of its
// loads before the first reduction, so enough bytes are in flight to stream
// at the copy rate.
constexpr int kDeltaRows = 8;  // rows per warp: 2 per pass (one per half-warp), 4 passes
template <bool kBF16>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const BackwardParams p) {
  using T = typename std::conditional<kBF16, __nv_bfloat16, __half>::type;
  constexpr int kPasses = kDeltaRows / 2;
  const long long rows = static_cast<long long>(p.B) * p.H * p.S_q;
  const int lane = threadIdx.x % 32, half = lane / 16, l16 = lane % 16;
  const long long row0 = (static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32) * kDeltaRows;
  uint4 a[kPasses], g[kPasses];
#pragma unroll
  for (int k = 0; k < kPasses; ++k) {
    const long long row = row0 + 2 * k + half;
    a[k] = g[k] = make_uint4(0u, 0u, 0u, 0u);
    if (row < rows) {
      const int i = static_cast<int>(row % p.S_q);
      const int bh = static_cast<int>(row / p.S_q);
      const int b = bh / p.H, h = bh % p.H;
      const size_t off = (p.bshd ? ((static_cast<size_t>(b) * p.S_q + i) * p.H + h) * kT
                                 : static_cast<size_t>(row) * kT) + l16 * 8;
      a[k] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.o) + off));
      g[k] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.dout) + off));
    }
  }
#pragma unroll
  for (int k = 0; k < kPasses; ++k) {
    const T* av = reinterpret_cast<const T*>(&a[k]);
    const T* gv = reinterpret_cast<const T*>(&g[k]);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) s = fmaf(static_cast<float>(av[e]), static_cast<float>(gv[e]), s);
#pragma unroll
    for (int m = 8; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);  // within the half
    const long long row = row0 + 2 * k + half;
    if (l16 == 0 && row < rows) p.delta[row] = s;
  }
}

// ---------------------------------------------------------------- dK / dV

template <bool kBF16>
__global__ void __launch_bounds__(kThreadsB, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dk,
                    const __grid_constant__ CUtensorMap tm_dv, const BackwardParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* s_k = smem;
  uint8_t* s_v = smem + kTile;
  float* s_rows = reinterpret_cast<float*>(smem + kOffRows);  // [stage][lse2 | delta][128]
  BwdCtl* ctl = reinterpret_cast<BwdCtl*>(smem + kOffCtl);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const int nkt = (p.S_kv + kT - 1) / kT;
  const int bh = blockIdx.x / nkt;
  const int kt = blockIdx.x % nkt;
  const int b = bh / p.H, h = bh % p.H;
  const int key0 = kt * kT;
  const int off = p.S_kv - p.S_q;  // bottom-right causal offset
  const int nqt = (p.S_q + kT - 1) / kT;
  // Query tiles that see any key of this tile: rows i >= key0 - off (causal).
  int first = 0;
  if (p.causal) first = max(0, key0 - off) / kT;
  const int n_steps = (p.causal && key0 - off > p.S_q - 1) ? 0 : nqt - first;

  if (warp == kWarpMmaB) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&ctl->res_full, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&ctl->full[s], 2);  // TMA bytes + the row statistics
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->s_full, 1);
    mbar_init(&ctl->dp_full, 1);
    mbar_init(&ctl->p_ready, kEwWarps);
    mbar_init(&ctl->ew_done, kEwWarps);
    mbar_init(&ctl->mma_done, 1);
    mbar_init(&ctl->tmem_free, kEwWarps);
    ctl->abort = 0;
    fence_mbar_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort;

  if (warp >= kEwWarps) {
   setmaxnreg_dec<kRegsCtl>();
   if (warp == kWarpLoad) {
    // ---------------------------------------------------------- producer
    if (n_steps > 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&ctl->res_full, 2 * kTile);
        load_tile(s_k, &tm_k, &ctl->res_full, key0, h, b, p.bshd);
        load_tile(s_v, &tm_v, &ctl->res_full, key0, h, b, p.bshd);
      }
      int issued = 0;
      for (int s = 0; s < n_steps; ++s) {
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        const int st = s % kRing;
        const int q0 = (first + s) * kT;
        // The tile's row statistics: every global load of a lane is issued
        // before any shared-memory store (a store between them, which the
        // compiler cannot prove distinct from the next load, serialised eight
        // memory round trips: ~7000 cycles per step, measured on GB300), and
        // before the wait for a free stage, so their latency overlaps it.
        const float* lse_b = p.lse + static_cast<size_t>(bh) * p.S_q;
        const float* dlt_b = p.delta + static_cast<size_t>(bh) * p.S_q;
        float lv[kT / 32], dv[kT / 32];
#pragma unroll
        for (int k = 0; k < kT / 32; ++k) {
          const int i = q0 + lane + 32 * k;
          lv[k] = i < p.S_q ? __ldg(lse_b + i) : 0.f;
          dv[k] = i < p.S_q ? __ldg(dlt_b + i) : 0.f;
        }
        bool ok = true;
        if (lane == 0 && s >= kRing)
          ok = mbar_wait(&ctl->empty[st], (s / kRing - 1) & 1, p.wait_limit_ns, p.err, 60);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        uint8_t* stage = smem + kOffRing + st * 2 * kTile;
        if (lane == 0) {
          mbar_arrive_expect_tx(&ctl->full[st], 2 * kTile);
          load_tile(stage, &tm_q, &ctl->full[st], q0, h, b, p.bshd);
          load_tile(stage + kTile, &tm_do, &ctl->full[st], q0, h, b, p.bshd);
        }
        float* rows = s_rows + st * 2 * kT;
#pragma unroll
        for (int k = 0; k < kT / 32; ++k) {
          rows[lane + 32 * k] = lv[k] * kLog2e;
          rows[kT + lane + 32 * k] = dv[k];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->full[st]);
        issued = s + 1;
      }
      if (lane == 0) {  // no copy may still be landing when the CTA exits
        for (int s = max(0, issued - kRing); s < issued; ++s)
          mbar_wait(&ctl->full[s % kRing], (s / kRing) & 1, p.wait_limit_ns, p.err, 61);
        mbar_wait(&ctl->res_full, 0, p.wait_limit_ns, p.err, 62);
      }
    }
    __syncwarp();
   } else if (warp == kWarpMmaB) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && n_steps > 0) {
      constexpr uint32_t id_s = idesc_f16(kBF16, kT, kT, false, false);
      constexpr uint32_t id_o = idesc_f16(kBF16, kT, kT, false, true);
      const uint32_t hi = sdesc_hi_sw128(1024);
      const uint32_t k_lo = sdesc_lo(smem_u32(s_k), 16);
      const uint32_t v_lo = sdesc_lo(smem_u32(s_v), 16);
      bool ok = mbar_wait(&ctl->res_full, 0, p.wait_limit_ns, p.err, 63);
      auto stage_of = [&](int s) { return smem_u32(smem + kOffRing + (s % kRing) * 2 * kTile); };
      auto wait_stage = [&](int s) {
        const bool w = mbar_wait(&ctl->full[s % kRing], (s / kRing) & 1, p.wait_limit_ns, p.err, 64);
        tc_fence_after_sync();
        return w;
      };
      // Step s: S^T_s = K Q_s^T into [0, 128) (signalled on s_full), dP^T_s = V
      // dO_s^T into [128, 256) (dp_full); dV += P^T_s dO_s once P^T is in place,
      // dK += dS^T_s Q_s once dS^T is (the walking tiles read MN-major).  S^T_{s+1}
      // follows dV_s, which has read P^T_s from S's columns, and dP^T_{s+1}
      // follows dK_s, which has read dS^T_s from dP's columns: the element-wise
      // warps start P^T_{s+1} from S^T_{s+1} alone while the tensor core runs
      // dK_s and dP^T_{s+1}.
      if (ok && (ok = wait_stage(0))) {
        mma_abt(tmem + 0, k_lo, sdesc_lo(stage_of(0), 16), hi, id_s);
        mma_commit(&ctl->s_full);
        mma_abt(tmem + 128, v_lo, sdesc_lo(stage_of(0) + kTile, 16), hi, id_s);
        mma_commit(&ctl->dp_full);
      }
      for (int s = 0; s < n_steps && ok; ++s) {
        const uint32_t stage = stage_of(s);
        const bool next = s + 1 < n_steps;
        if (!(ok = mbar_wait(&ctl->p_ready, s & 1, p.wait_limit_ns, p.err, 68))) break;
        tc_fence_after_sync();
        mma_tmem_a_split(tmem + 256, tmem + 0, sdesc_lo(stage + kTile, kPanel), hi, id_o, s > 0);
        // S^T_{s+1} goes first if its tiles have landed (a non-blocking test):
        // waiting for them here would hold back dK_s.
        bool s_next = false;
        if (next && mbar_test_wait(&ctl->full[(s + 1) % kRing], ((s + 1) / kRing) & 1)) {
          tc_fence_after_sync();
          mma_abt(tmem + 0, k_lo, sdesc_lo(stage_of(s + 1), 16), hi, id_s);
          mma_commit(&ctl->s_full);
          s_next = true;
        }
        if (!(ok = mbar_wait(&ctl->ew_done, s & 1, p.wait_limit_ns, p.err, 65))) break;
        tc_fence_after_sync();
        mma_tmem_a_split(tmem + 384, tmem + 128, sdesc_lo(stage, kPanel), hi, id_o, s > 0);
        mma_commit(&ctl->empty[s % kRing]);
        if (next) {
          if (!s_next) {
            if (!(ok = wait_stage(s + 1))) break;
            mma_abt(tmem + 0, k_lo, sdesc_lo(stage_of(s + 1), 16), hi, id_s);
            mma_commit(&ctl->s_full);
          }
          mma_abt(tmem + 128, v_lo, sdesc_lo(stage_of(s + 1) + kTile, 16), hi, id_s);
          mma_commit(&ctl->dp_full);
        }
      }
      if (!ok) *abort_flag = 1;
      mma_commit(&ctl->mma_done);
      mbar_wait(&ctl->mma_done, 0, p.wait_limit_ns, p.err, 66);
    }
    __syncwarp();
    mbar_wait(&ctl->tmem_free, 0, p.wait_limit_ns, p.err, 67);
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
   }
  } else {
    setmaxnreg_inc<kRegsEw>();
    // ---------------------------------------------------------- element-wise
    const int g = warp / 4;                // column group of this warp
    const int r = (warp % 4) * 32 + lane;  // key row within the tile
    const int key = key0 + r;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    bool ok = true;
    for (int s = 0; s < n_steps; ++s) {
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->s_full, s & 1, p.wait_limit_ns, p.err, 70));
      if (!ok) break;
      tc_fence_after_sync();
      const int st = s % kRing;
      const float* lse2 = s_rows + st * 2 * kT;
      const float* dlt = lse2 + kT;
      const int q0 = (first + s) * kT;
      const bool full = key0 + kT <= p.S_kv && q0 + kT <= p.S_q &&
                        (!p.causal || key0 + kT - 1 <= q0 + off);
      auto lse2_of = [=](int col) { return *reinterpret_cast<const float2*>(lse2 + col); };
      auto delta_of = [=](int col) { return *reinterpret_cast<const float2*>(dlt + col); };
      auto visible = [=](int col) {
        const int i = q0 + col;
        return key < p.S_kv && i < p.S_q && (!p.causal || key <= i + off);
      };
      if (full)
        ok = elementwise_step_p_first<kBF16, false>(lane_addr, g, 0, 128, p.scale_log2, lse2_of,
                                                    delta_of, visible, &ctl->p_ready,
                                                    &ctl->dp_full, s & 1, p.wait_limit_ns, p.err,
                                                    lane);
      else
        ok = elementwise_step_p_first<kBF16, true>(lane_addr, g, 0, 128, p.scale_log2, lse2_of,
                                                   delta_of, visible, &ctl->p_ready,
                                                   &ctl->dp_full, s & 1, p.wait_limit_ns, p.err,
                                                   lane);
      if (!ok) break;
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->ew_done);
    }
    // ---------------------------------------------------------- epilogue
    if (ok && n_steps > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->mma_done, 0, p.wait_limit_ns, p.err, 71));
    tc_fence_after_sync();
    const bool have = ok && n_steps > 0;
    // dV into the V tile (group 0), dK times scale into the K tile (group 1):
    // both tiles are dead.
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t o[64] = {};
      if (have) tmem_ld64_wait(lane_addr + 256 + 128 * g + hh * 64, o);
      stage_row<kBF16>(g == 0 ? s_v : s_k, r, hh, o, g == 0 ? 1.f : p.scale);
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->tmem_free);
    fence_proxy_async_smem();
    named_barrier_sync(1, kEwWarps * 32);
    if (threadIdx.x == 0) {
      store_tile(&tm_dv, s_v, key0, h, b, p.bshd);
      store_tile(&tm_dk, s_k, key0, h, b, p.bshd);
      tma_store_commit();
      tma_store_wait_all();
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- dQ

// The dQ kernel streams K and V through rings of their own: V_j is read only
// by dP_j and is released early; K_j is read by S_j and, one step later in
// the pipeline below, by dQ += dS_j K_j.  Three K stages and two V stages of
// 32 KB fit beside the resident Q and dO.
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kOffDqK = 2 * kTile;
constexpr int kOffDqV = kOffDqK + kKStages * kTile;
constexpr int kOffDqCtl = kOffDqV + kVStages * kTile;
constexpr int kSmemDq = kOffDqCtl + 256 + 1024;

struct DqCtl {
  uint64_t res_full;            // the resident Q and dO have landed
  uint64_t k_full[kKStages];    // K_j has landed
  uint64_t k_empty[kKStages];   // S_j and dQ_j have read K_j
  uint64_t v_full[kVStages];
  uint64_t v_empty[kVStages];   // dP_j has read V_j
  uint64_t mm_full;             // S_j and dP_j are in tensor memory
  uint64_t loaded;              // the element-wise warps hold S_j and dP_j in registers
  uint64_t ew_done;             // dS_j is in tensor memory (columns [384, 448))
  uint64_t ds_free;             // dQ_{j-1} has read the dS columns
  uint64_t mma_done;            // every MMA of the CTA has completed
  uint64_t tmem_free;           // the element-wise warps are done with tensor memory
  uint64_t prod_done;           // warp 9's last products have completed
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DqCtl) <= 256, "control block must fit its reserved bytes");
static_assert(kSmemDq <= 232448, "dQ shared memory exceeds the per-block limit");

// Pipelined per key tile j: S_j = Q K_j^T and dP_j = dO V_j^T into tensor
// memory [0, 256); the element-wise warps load both into registers and
// announce it, so the MMA warp issues S_{j+1}, dP_{j+1} over them while dS_j
// is computed and stored in columns [384, 448) of its own; then dQ += dS_j K_j
// into [256, 384).
template <bool kBF16>
__global__ void __launch_bounds__(kThreadsB, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const BackwardParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* s_q = smem;
  uint8_t* s_do = smem + kTile;
  uint8_t* s_k = smem + kOffDqK;  // kKStages tiles
  uint8_t* s_v = smem + kOffDqV;  // kVStages tiles
  DqCtl* ctl = reinterpret_cast<DqCtl*>(smem + kOffDqCtl);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const int nqt = (p.S_q + kT - 1) / kT;
  const int bh = blockIdx.x / nqt;
  const int qt = blockIdx.x % nqt;
  const int b = bh / p.H, h = bh % p.H;
  const int q0 = qt * kT;
  const int off = p.S_kv - p.S_q;
  int keys = p.S_kv;
  if (p.causal) keys = min(keys, min(q0 + kT, p.S_q) - 1 + off + 1);
  const int n_steps = keys <= 0 ? 0 : (keys + kT - 1) / kT;

  if (warp == kWarpMmaB) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&ctl->res_full, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], 1);
    }
    mbar_init(&ctl->mm_full, 1);
    mbar_init(&ctl->loaded, kEwWarps);
    mbar_init(&ctl->ew_done, kEwWarps);
    mbar_init(&ctl->ds_free, 1);
    mbar_init(&ctl->mma_done, 1);
    mbar_init(&ctl->tmem_free, kEwWarps);
    mbar_init(&ctl->prod_done, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort;

  if (warp >= kEwWarps) {
   setmaxnreg_dec<kRegsCtl>();
   if (warp == kWarpLoad) {
    // ---------------------------------------------------------- producer
    if (lane == 0 && n_steps > 0) {
      mbar_arrive_expect_tx(&ctl->res_full, 2 * kTile);
      load_tile(s_q, &tm_q, &ctl->res_full, q0, h, b, p.bshd);
      load_tile(s_do, &tm_do, &ctl->res_full, q0, h, b, p.bshd);
      int issued = 0, v_issued = 0;  // K and V tiles whose copies were issued
      for (int s = 0; s < n_steps && !*abort_flag; ++s) {
        const int sk = s % kKStages, sv = s % kVStages;
        if (s >= kKStages &&
            !mbar_wait(&ctl->k_empty[sk], (s / kKStages - 1) & 1, p.wait_limit_ns, p.err, 80)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&ctl->k_full[sk], kTile);
        load_tile(s_k + sk * kTile, &tm_k, &ctl->k_full[sk], s * kT, h, b, p.bshd);
        issued = s + 1;  // K_s is in flight from here on
        if (s >= kVStages &&
            !mbar_wait(&ctl->v_empty[sv], (s / kVStages - 1) & 1, p.wait_limit_ns, p.err, 79)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&ctl->v_full[sv], kTile);
        load_tile(s_v + sv * kTile, &tm_v, &ctl->v_full[sv], s * kT, h, b, p.bshd);
        v_issued = s + 1;
      }
      // No copy may still be landing when the CTA exits: wait (bounded) for
      // the last load issued into every stage.
      for (int s = max(0, issued - kKStages); s < issued; ++s)
        mbar_wait(&ctl->k_full[s % kKStages], (s / kKStages) & 1, p.wait_limit_ns, p.err, 81);
      for (int s = max(0, v_issued - kVStages); s < v_issued; ++s)
        mbar_wait(&ctl->v_full[s % kVStages], (s / kVStages) & 1, p.wait_limit_ns, p.err, 78);
      mbar_wait(&ctl->res_full, 0, p.wait_limit_ns, p.err, 82);
    }
    __syncwarp();
   } else if (warp == kWarpMmaB) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && n_steps > 0) {
      constexpr uint32_t id_s = idesc_f16(kBF16, kT, kT, false, false);
      constexpr uint32_t id_o = idesc_f16(kBF16, kT, kT, false, true);
      const uint32_t hi = sdesc_hi_sw128(1024);
      const uint32_t q_lo = sdesc_lo(smem_u32(s_q), 16);
      const uint32_t do_lo = sdesc_lo(smem_u32(s_do), 16);
      // S_s = Q K_s^T and dP_s = dO V_s^T; V_s is released right after.
      auto products = [&](int s) {
        const int sk = s % kKStages, sv = s % kVStages;
        if (!mbar_wait(&ctl->k_full[sk], (s / kKStages) & 1, p.wait_limit_ns, p.err, 84) ||
            !mbar_wait(&ctl->v_full[sv], (s / kVStages) & 1, p.wait_limit_ns, p.err, 89))
          return false;
        tc_fence_after_sync();
        mma_abt(tmem + 0, q_lo, sdesc_lo(smem_u32(s_k + sk * kTile), 16), hi, id_s);
        mma_abt(tmem + 128, do_lo, sdesc_lo(smem_u32(s_v + sv * kTile), 16), hi, id_s);
        mma_commit(&ctl->mm_full);
        mma_commit(&ctl->v_empty[sv]);
        return true;
      };
      // This thread issues the products; dQ += dS_s K_s comes from warp 10's
      // thread, so the two threads' waits and commits overlap instead of
      // adding up.  They touch different tensor-memory columns and are
      // ordered only through the element-wise warps' barriers.
      bool ok = mbar_wait(&ctl->res_full, 0, p.wait_limit_ns, p.err, 83);
      if (ok) ok = products(0);
      for (int s = 0; s + 1 < n_steps && ok; ++s) {
        if (!(ok = mbar_wait(&ctl->loaded, s & 1, p.wait_limit_ns, p.err, 88))) break;
        ok = products(s + 1);
      }
      if (!ok) *abort_flag = 1;
      mma_commit(&ctl->prod_done);
      mbar_wait(&ctl->prod_done, 0, p.wait_limit_ns, p.err, 86);
    }
    __syncwarp();
    mbar_wait(&ctl->tmem_free, 0, p.wait_limit_ns, p.err, 87);
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
   } else if (warp == kWarpMmaDq) {
    // ---------------------------------------------------------- dQ issuer
    if (lane == 0 && n_steps > 0) {
      constexpr uint32_t id_o = idesc_f16(kBF16, kT, kT, false, true);
      const uint32_t hi = sdesc_hi_sw128(1024);
      bool ok = true;
      for (int s = 0; s < n_steps && ok; ++s) {
        if (!(ok = mbar_wait(&ctl->ew_done, s & 1, p.wait_limit_ns, p.err, 85))) break;
        tc_fence_after_sync();
        // dQ += dS_s K_s (dS in columns [384, 448)), K read MN-major
        const int sk = s % kKStages;
        mma_tmem_a(tmem + 256, tmem + 384, sdesc_lo(smem_u32(s_k + sk * kTile), kPanel), hi, id_o,
                   s > 0);
        mma_commit(&ctl->ds_free);
        mma_commit(&ctl->k_empty[sk]);  // S_s (warp 9) completed before dS_s was published
      }
      if (!ok) *abort_flag = 1;
      // The last MMAs of the CTA: every product came before the last dS.
      mma_commit(&ctl->mma_done);
      mbar_wait(&ctl->mma_done, 0, p.wait_limit_ns, p.err, 77);
    }
    __syncwarp();
   }
  } else {
    setmaxnreg_inc<kRegsEw>();
    // ---------------------------------------------------------- element-wise
    const int g = warp / 4;                // column group of this warp
    const int r = (warp % 4) * 32 + lane;  // query row within the tile
    const int i = q0 + r;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    const size_t ridx = static_cast<size_t>(bh) * p.S_q + i;
    const float lse2 = i < p.S_q ? p.lse[ridx] * kLog2e : 0.f;
    const float dlt = i < p.S_q ? p.delta[ridx] : 0.f;
    const float c = p.scale_log2;
    bool ok = true;
    for (int s = 0; s < n_steps; ++s) {
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->mm_full, s & 1, p.wait_limit_ns, p.err, 90));
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t x[64], y[64];
      tmem_ld64_wait(lane_addr + 0 + 64 * g, x);    // S, this warp's 64 key columns
      tmem_ld64_wait(lane_addr + 128 + 64 * g, y);  // dP
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->loaded);  // the MMA warp may overwrite S and dP
      const int k0 = s * kT;
      const bool full = k0 + kT <= p.S_kv && q0 + kT <= p.S_q &&
                        (!p.causal || k0 + kT - 1 <= q0 + off);
      uint32_t dd[32];  // dS as 16-bit pairs: column 32g + q holds keys 64g + 2q, + 1
      // Column pairs in packed fp32 (f32x2): one instruction per two elements.
      const uint64_t c2 = f2_pack(c, c), nl2 = f2_pack(-lse2, -lse2);
      const uint64_t nd2 = f2_pack(-dlt, -dlt), z2 = f2_pack(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        float a0, a1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(x[2 * q]), __uint_as_float(x[2 * q + 1])), c2,
                         nl2),
                  a0, a1);
        float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
        if (!full) {
          const int key = k0 + 64 * g + 2 * q;
          const bool row_ok = i < p.S_q;
          p0 = (row_ok && key < p.S_kv && (!p.causal || key <= i + off)) ? p0 : 0.f;
          p1 = (row_ok && key + 1 < p.S_kv && (!p.causal || key + 1 <= i + off)) ? p1 : 0.f;
        }
        const uint64_t t =
            f2_add(f2_pack(__uint_as_float(y[2 * q]), __uint_as_float(y[2 * q + 1])), nd2);
        float d0, d1;
        f2_unpack(f2_fma(f2_pack(p0, p1), t, z2), d0, d1);
        dd[q] = pack2<kBF16>(d0, d1);
      }
      // dQ_{s-1} must have read the dS columns before they are overwritten.
      if (s > 0) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&ctl->ds_free, (s - 1) & 1, p.wait_limit_ns, p.err, 92));
        if (!ok) break;
        tc_fence_after_sync();
      }
      tmem_st16(lane_addr + 384 + 32 * g, *reinterpret_cast<uint32_t(*)[16]>(dd));
      tmem_st16(lane_addr + 384 + 32 * g + 16, *reinterpret_cast<uint32_t(*)[16]>(dd + 16));
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->ew_done);
    }
    if (ok && n_steps > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->mma_done, 0, p.wait_limit_ns, p.err, 91));
    tc_fence_after_sync();
    const bool have = ok && n_steps > 0;
    {  // dQ times scale into the Q tile (dead now): columns [64g, 64g + 64)
      uint32_t o[64] = {};
      if (have) tmem_ld64_wait(lane_addr + 256 + g * 64, o);
      stage_row<kBF16>(s_q, r, g, o, p.scale);
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->tmem_free);
    fence_proxy_async_smem();
    named_barrier_sync(1, kEwWarps * 32);
    if (threadIdx.x == 0) {
      store_tile(&tm_dq, s_q, q0, h, b, p.bshd);
      tma_store_commit();
      tma_store_wait_all();
    }
    __syncwarp();
  }
}

template <class K>
cudaError_t configure(K kern, int smem_bytes) {
  // The in-kernel register split assumes exactly kRegsLaunchB registers per
  // thread at launch; with fewer, setmaxnreg.inc would never complete.
  cudaFuncAttributes fa{};
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kRegsLaunchB) return cudaErrorInvalidConfiguration;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

template <bool kBF16>
cudaError_t launch_all(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& dout, const CUtensorMap& dq, const CUtensorMap& dk,
                       const CUtensorMap& dv, const BackwardParams& p, cudaStream_t stream) {
  static std::atomic<unsigned long long> configured{0};  // per template instance, per device
  cudaError_t ce = attn_host::once_per_device(configured, [&]() {
    cudaError_t e = configure(bwd_dkdv_kernel<kBF16>, kSmemB);
    return e == cudaSuccess ? configure(bwd_dq_kernel<kBF16>, kSmemDq) : e;
  });
  if (ce != cudaSuccess) return ce;
  const long long rows = static_cast<long long>(p.B) * p.H * p.S_q;
  if (rows > 0) {
    bwd_delta_kernel<kBF16><<<static_cast<unsigned>((rows + 8 * kDeltaRows - 1) / (8 * kDeltaRows)),
                              256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int nkt = (p.S_kv + kT - 1) / kT;
  const int nqt = (p.S_q + kT - 1) / kT;
  if (p.B * p.H * nkt > 0)
    bwd_dkdv_kernel<kBF16><<<p.B * p.H * nkt, kThreadsB, kSmemB, stream>>>(q, k, v, dout, dk,
                                                                           dv, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.B * p.H * nqt > 0)
    bwd_dq_kernel<kBF16><<<p.B * p.H * nqt, kThreadsB, kSmemDq, stream>>>(q, k, v, dout, dq, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t backward_launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dout, const CUtensorMap& dq, const CUtensorMap& dk,
                            const CUtensorMap& dv, const BackwardParams& p, bool bf16,
                            cudaStream_t stream) {
  return bf16 ? launch_all<true>(q, k, v, dout, dq, dk, dv, p, stream)
              : launch_all<false>(q, k, v, dout, dq, dk, dv, p, stream);
}

}  // namespace attn_sm103a
