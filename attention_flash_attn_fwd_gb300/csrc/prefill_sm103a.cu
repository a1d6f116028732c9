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
//    diagonal tiles are masked element by element;
//  * contiguous forms run persistent CTAs (one per SM) that take (batch,
//    head, query block) units from a per-stream counter in launch order, so
//    the units in flight are consecutive (their heads' K/V stay in L2) and
//    faster CTAs take more of the unequal causal units.  Between units nothing
//    drains: Q_t is refilled once the unit's last S MMA of tile t has read it,
//    K/V keep streaming through the same ring, the next unit's first S MMAs
//    run during the epilogue, and O leaves without touching Q's tiles (which
//    already hold the next unit): by TMA store from staging tiles of its own
//    where shared memory has room (FP8, D = 64), else in whole-sector stores
//    straight from registers.  Measured on
//    GB300, the one-unit CTAs spent ~5.8 us per unit outside the main loop
//    (set-up, the first Q/K tiles arriving, epilogue, CTA turnover).
//
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D),
// O1 [256+D, 256+2D).  P_t (16-bit pairs) overwrites the first 64 columns of
// S_t.
//
// The extend form (new tokens of a sequence against its cached keys, Wave
// February 2025 Release, "Extend Attention"; WAVE MLSys 2026 summary,
// Integration: SGLang extend) is the same kernel with kPaged: the whole TMA
// warp gathers each 128-key K/V tile page by page through the page table
// (one lane per page-sized box), the key count and the causal diagonal come
// from the sequence's kv_len, and query head h reads kv head h / group.
// Every box costs the TMA unit a fixed overhead, so with small pages the
// paged path issues no L2 prefetch boxes (measured on GB300 with 16-token
// pages: 1.62 ms with them, 0.97 ms without, for the same loads), and for
// pages of at most 16 keys two CTAs share the box work: a cluster of 2 holds
// query heads 2k and 2k+1 of one kv head and one query block, each CTA
// issues every other page box multicast to both, and each MMA warp releases
// a K/V stage in both CTAs (0.96 -> 0.80 ms with 16-token pages).
//
// The FP8 form (kFp8; Wave February 2025 Release, EvoFormer list, "FAv3 -
// FP8") reads E4M3 Q, K, V: tiles are half the bytes (one 128-byte swizzled
// panel holds a 128-wide row), both products run as `.kind::f8f6f4` MMAs (K = 32 per
// instruction), P is written to tensor memory as E4M3 (four per column) and
// the per-tensor descale factors fold into the softmax scale and the final
// 1/l.  O (bf16 or fp16) is staged in its own shared-memory tiles.
#include "prefill_sm103a.h"

#include "host_once.h"
#include "sm103a_ptx.cuh"

namespace attn_sm103a {

namespace {

constexpr int kBM = 128;      // query rows per tile
constexpr int kBN = 128;      // keys per KV tile
constexpr int kTiles = 2;     // query tiles per CTA
constexpr int kThreads = 384; // 2 softmax warpgroups + 1 warpgroup {TMA, MMA, 2 idle}
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
// Registers are granted per warpgroup: 384 threads launch with 168 each
// (64512 in all).  The softmax warpgroups take 216, the TMA/MMA warpgroup
// keeps 72 (its unit loop spills below that): 2*128*216 + 128*72 = 64512,
// exactly the launch total.
constexpr int kRegsAtLaunch = 168;
constexpr int kRegsSoftmax = 216;
constexpr int kRegsControl = 72;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsControl <= kThreads * kRegsAtLaunch,
              "register split exceeds the block's launch allocation");
constexpr float kRescaleThreshold = 8.0f;  // log2 units

constexpr int kCtlBytesFwd = 512;  // reserved for SharedCtl (checked below)

template <int D, bool kFp8 = false, bool kPaged = false>
struct Cfg {
  static constexpr int kElt = kFp8 ? 1 : 2;               // bytes per Q/K/V element
  static constexpr int kTileBytes = kBM * D * kElt;       // one Q/K/V tile
  static constexpr int kOTileBytes = kBM * D * 2;         // one O tile (16-bit)
  static constexpr int kBoxCols = 128 / kElt;             // columns per 128-byte TMA box
  static constexpr int kBoxes = D / kBoxCols;             // boxes (swizzle panels) per row
  static constexpr int kKeysPerPV = 32 / kElt;            // keys per PV MMA instruction
  static constexpr int kStages = kFp8 ? 8 : ((D == 128) ? 5 : 10);  // KV ring depth
  // O leaves the contiguous forms by TMA store from staging tiles of their own
  // where shared memory has room for them (FP8, D = 64); at D = 128 in 16
  // bits the 5-stage ring fills shared memory and O is stored straight from
  // registers (measured faster there than staging with a shallower ring).
  static constexpr bool kStagedO = !kPaged && (kFp8 || D == 64);
  static constexpr int kOStageOff = kTiles * kTileBytes + kStages * kTileBytes;
  static constexpr int kSmemData = kOStageOff + (kStagedO ? kTiles * kOTileBytes : 0);
  static constexpr int kSmemBytes = kSmemData + 1024 /*align*/ + kCtlBytesFwd;
  // tensor-memory columns of S_t and O_t
  __device__ static constexpr uint32_t col_s(int t) { return t * 128u; }
  __device__ static constexpr uint32_t col_o(int t) { return 256u + t * D; }
};

struct SharedCtl {
  uint64_t q_full[kTiles];
  uint64_t q_empty[kTiles];    // the unit's last S MMA of tile t has read Q_t
  uint64_t s_full[kTiles];
  uint64_t p_full[kTiles];     // P_t (all 128 keys) is in tensor memory
  uint64_t o_full[kTiles];     // the unit's last PV MMA of tile t is done (tiles with keys)
  uint64_t o_free[kTiles];     // the softmax warps of tile t hold O_t in registers
  uint64_t unit_full[2];       // a unit id was published in unit_ring
  uint64_t unit_empty[2];      // the MMA warp and every softmax warp read it
  uint64_t tmem_free;  // every softmax warp is done reading tensor memory
  uint64_t kv_full[10];
  uint64_t kv_empty[10];
  uint64_t tail_v;     // extend form: the V tile holding the sequence end has landed
  int unit_ring[2];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(SharedCtl) <= kCtlBytesFwd, "control block must fit its reserved bytes");

// TMA load of one 64-column box of rows [row, row + 128) of (batch b, head h).
// BHSD maps are (D, S, H, B); BSHD maps are (D, H, S, B).
__device__ __forceinline__ void load_box(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                         int row, int h, int b, int bshd) {
  if (bshd)
    tma_load_4d(dst, map, bar, x, h, row, b);
  else
    tma_load_4d(dst, map, bar, x, row, h, b);
}

// L2 prefetch of one 64-column box (same coordinates as load_box).
__device__ __forceinline__ void prefetch_box(const CUtensorMap* map, int x, int row, int h, int b,
                                             int bshd) {
  if (bshd)
    tma_prefetch_l2_4d(map, x, h, row, b);
  else
    tma_prefetch_l2_4d(map, x, row, h, b);
}

// KV tiles the producer prefetches into L2 ahead of its shared-memory loads.
// The CTAs of one (batch, head) stream the same K/V tiles at about the same
// time, so without it every tile load waits for a DRAM round trip.
constexpr int kL2PrefetchTiles = 4;

// Number of KV tiles a query tile [row0, row0 + kBM) must visit.
__device__ __forceinline__ int kv_tiles_for(int row0, int S_kv, const PrefillParams& p) {
  int keys = S_kv;
  if (p.causal) {
    int last_row = min(row0 + kBM, p.S_q) - 1;
    keys = min(keys, last_row + (S_kv - p.S_q) + 1);
  }
  return keys <= 0 ? 0 : (keys + kBN - 1) / kBN;
}

// Producer of the extend form: the whole warp streams K/V tiles gathered
// through the page table.  Lane (bx, half) owns box bx (one page, or 128 rows
// of a larger page) of 64-column half `half` of each tile.  The pool is seen
// as a 2-D tensor: rows are (page, slot), columns (kv head, d).  In a CTA
// pair (cs == 2) this CTA issues the boxes with bx % 2 == rank, multicast to
// both; each CTA still expects the whole tile on its own barrier.  Keys past the
// sequence end are never multiplied by a nonzero weight, but their V rows
// may hold anything (0 * NaN = NaN), so the V tile holding the sequence end
// lands on its own barrier, the warp zeroes rows [valid, 128) and only then
// publishes the stage.
template <int D>
__device__ __forceinline__ void produce_paged(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                              const CUtensorMap& tm_v, const PrefillParams& p,
                                              SharedCtl* ctl, uint8_t* s_q, uint8_t* s_kv, int b,
                                              int h, int S_kv, int row_base, int n_all,
                                              int lane, int cs, int rank) {
  using C = Cfg<D>;
  constexpr int kHalves = D / 64;
  constexpr uint32_t kAll = 0xffffffffu;
  const int g = h / p.group;
  const int ps = p.page_size;
  const int box_rows = min(ps, kBN);
  const int half = lane % kHalves;
  const int bx = lane / kHalves;
  const int32_t* pt = p.page_table + static_cast<size_t>(b) * p.max_pages;
  // Pool row of this lane's box in KV tile j; false if the box holds no key.
  // A page id outside the pool is flagged and replaced by the row just past
  // the pool's end, where the TMA fills the box with zeros.
  auto locate = [&](int j, int& row) {
    const int key = j * kBN + bx * box_rows;
    if (bx * box_rows >= kBN || key >= S_kv) return false;
    int page = __ldg(pt + key / ps);
    if (page < 0 || page >= p.num_pages) {
      record_error(p.err, kErrBadArgument, 4);
      page = p.num_pages;
    }
    row = page * ps + key % ps;
    return true;
  };
  volatile int* abort_flag = &ctl->abort;
  if (lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
    for (int t = 0; t < kTiles; ++t) {
      mbar_arrive_expect_tx(&ctl->q_full[t], C::kTileBytes);
      for (int x = 0; x < kHalves; ++x)
        tma_load_4d(s_q + t * C::kTileBytes + x * (kBM * 128), &tm_q, &ctl->q_full[t], x * 64, h,
                    row_base + t * kBM, b);
    }
  }
  int issued = 0, tail_idx = -1;
  for (int j = 0; j < n_all; ++j) {
    if (__shfl_sync(kAll, *abort_flag, 0)) break;
    int prow = 0;
    const bool mine = locate(j, prow);
    const int valid = min(kBN, S_kv - j * kBN);  // keys of this tile inside the sequence
    const int n_box = (valid + box_rows - 1) / box_rows;
    const uint32_t bytes = static_cast<uint32_t>(n_box * box_rows * 128 * kHalves);
    bool ok = true;
#pragma unroll 1
    for (int kind = 0; kind < 2 && ok; ++kind) {
      const int idx = 2 * j + kind;
      const int st = idx % C::kStages;
      const int round = idx / C::kStages;
      if (round > 0) {
        bool w = true;
        if (lane == 0) w = mbar_wait(&ctl->kv_empty[st], (round - 1) & 1, p.wait_limit_ns, p.err, 13);
        if (!(ok = __shfl_sync(kAll, w, 0))) break;
      }
      uint8_t* dst = s_kv + st * C::kTileBytes;
      const bool fix_v = kind == 1 && valid < kBN;
      uint64_t* bar = fix_v ? &ctl->tail_v : &ctl->kv_full[st];
      if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
      __syncwarp();
      if (mine) {
        uint8_t* box_dst = dst + half * (kBN * 128) + bx * box_rows * 128;
        const CUtensorMap* map = kind ? &tm_v : &tm_k;
        if (cs == 1)
          tma_load_2d(box_dst, map, bar, g * D + half * 64, prow);
        else if (bx % 2 == rank)
          tma_load_2d_multicast(box_dst, map, bar, g * D + half * 64, prow, 0x3);
      }
      issued = idx + 1;
      if (fix_v) {
        tail_idx = idx;
        if (!(ok = __all_sync(kAll, mbar_wait(&ctl->tail_v, 0, p.wait_limit_ns, p.err, 14))))
          break;
        const int chunks = (kBN - valid) * 8;  // 16-byte chunks past the end, per half
        for (int c = lane; c < chunks * kHalves; c += 32) {
          const int hh = c / chunks, rem = c % chunks;
          *reinterpret_cast<uint4*>(dst + hh * (kBN * 128) + (valid + rem / 8) * 128 +
                                    (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // the zeros must be visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->kv_full[st]);
      }
    }
    if (!ok) {
      if (lane == 0) *abort_flag = 1;
      break;
    }
  }
  // Never leave the CTA with a copy still landing in shared memory.
  if (lane == 0) {
    for (int idx = max(0, issued - C::kStages); idx < issued; ++idx)
      if (idx == tail_idx)
        mbar_wait(&ctl->tail_v, 0, p.wait_limit_ns, p.err, 15);
      else
        mbar_wait(&ctl->kv_full[idx % C::kStages], (idx / C::kStages) & 1, p.wait_limit_ns,
                  p.err, 11);
    for (int t = 0; t < kTiles; ++t) mbar_wait(&ctl->q_full[t], 0, p.wait_limit_ns, p.err, 12);
  }
}

// Keys of sequence b in the extend form: kv_lens[b], clamped to the page
// table's capacity (a value outside [0, capacity] is flagged).
__device__ __forceinline__ int extend_kv_len(int b, const PrefillParams& p) {
  const int cap = p.max_pages * p.page_size;
  int kv = p.kv_lens[b];
  if (kv < 0 || kv > cap) {
    if (threadIdx.x == 0) record_error(p.err, kErrBadArgument, 3);
    kv = kv < 0 ? 0 : cap;
  }
  return kv;
}

template <int D, bool kBF16, bool kPaged, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o, const PrefillParams p) {
  using C = Cfg<D, kFp8, kPaged>;
  extern __shared__ uint8_t smem_raw[];
  // Offset from the __shared__ array, so accesses stay in the shared space.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* s_q = smem;                                   // kTiles tiles
  uint8_t* s_kv = smem + kTiles * C::kTileBytes;         // kStages tiles
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + C::kSmemData);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // Work unit: (batch, head, 256-row query block), numbered head-major with
  // the longest causal block of a head first.  Without a scheduler counter a
  // CTA runs the one unit its index names; with one (p.sched, contiguous
  // form) a persistent CTA takes the next unit from it until none is left,
  // so the CTAs in flight always hold consecutive units: a few heads, whose
  // K/V stay in L2.
  const int nqb = p.num_q_blocks;
  // A CTA pair (cluster of 2, extend form only) holds query heads 2k, 2k+1.
  const int cs = (kPaged && p.pair) ? 2 : 1;
  const int rank = cs == 2 ? static_cast<int>(cluster_ctarank()) : 0;
  const int n_units = p.B * (p.H / cs) * nqb;
  const bool dyn = !kPaged && p.sched != nullptr;
  struct Unit {
    int b, h, S_kv, row_base, n_kv0, n_kv1, n_all;
    __device__ int n_kv(int t) const { return t == 0 ? n_kv0 : n_kv1; }
  };
  auto unit_info = [&](int u) {
    Unit U;
    const int bh = u / nqb;
    const int qb = nqb - 1 - (u % nqb);
    U.b = bh / (p.H / cs);
    U.h = (bh % (p.H / cs)) * cs + rank;
    U.S_kv = kPaged ? extend_kv_len(U.b, p) : p.S_kv;  // keys of this sequence
    U.row_base = qb * (kTiles * kBM);
    U.n_kv0 = kv_tiles_for(U.row_base, U.S_kv, p);
    U.n_kv1 = kv_tiles_for(U.row_base + kBM, U.S_kv, p);
    U.n_all = max(U.n_kv0, U.n_kv1);  // tile 1 never needs fewer than tile 0
    return U;
  };
  // Unit n of this CTA, published by the producer in unit_ring[n % 2]; -1 ends.
  auto read_unit = [&](int n) -> int {
    return *reinterpret_cast<volatile int*>(&ctl->unit_ring[n & 1]);
  };

  if (warp == kWarpMma) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&ctl->q_full[t], 1);
      mbar_init(&ctl->q_empty[t], 1);
      mbar_init(&ctl->s_full[t], 1);
      mbar_init(&ctl->p_full[t], 4);
      mbar_init(&ctl->o_full[t], 1);
      mbar_init(&ctl->o_free[t], 4);
    }
    for (int sl = 0; sl < 2; ++sl) {
      mbar_init(&ctl->unit_full[sl], 1);
      mbar_init(&ctl->unit_empty[sl], 1 + 8);  // the MMA warp and the 8 softmax warps
    }
    mbar_init(&ctl->tmem_free, 8);
    mbar_init(&ctl->tail_v, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&ctl->kv_full[s], 1);
      mbar_init(&ctl->kv_empty[s], cs);  // released by the MMA warp of every CTA of the pair
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  if (cs == 2) cluster_sync();  // the partner's barriers exist before any multicast
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort;

  if (warp >= 8) {
   // ============================================= control warpgroup
   setmaxnreg_dec<kRegsControl>();
   if (kPaged && warp == kWarpTma) {
    // ------------------------------------------------- producer (paged K/V)
    // One unit per CTA: publish it, stream it, then publish the end.
    const int u = static_cast<int>(blockIdx.x) / cs;
    if (lane == 0) {
      ctl->unit_ring[0] = u;
      mbar_arrive(&ctl->unit_full[0]);
    }
    // Q is loaded even when the unit has no key (the MMA warp waits for it).
    const Unit U = unit_info(u);
    produce_paged<D>(tm_q, tm_k, tm_v, p, ctl, s_q, s_kv, U.b, U.h, U.S_kv, U.row_base, U.n_all,
                     lane, cs, rank);
    if (lane == 0) {
      ctl->unit_ring[1] = -1;
      mbar_arrive(&ctl->unit_full[1]);
    }
    __syncwarp();
   } else if (warp == kWarpTma) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      int issued = 0;    // K/V loads issued, all units
      int q_loads = 0;   // units whose Q was loaded
      bool ok = true;
      // The producer runs ahead of the MMAs and waits for free stages most of
      // the time.  In the 16-bit forms it sleeps between tests, leaving the
      // issue slots of its scheduler to the softmax warps there (C3 ~1%
      // faster); with FP8's shorter steps the wake-up delay costs more.
      auto wait_free = [&](uint64_t* bar, uint32_t parity, int site) {
        return kFp8 ? mbar_wait(bar, parity, p.wait_limit_ns, p.err, site)
                    : mbar_wait_sleep(bar, parity, p.wait_limit_ns, p.err, site, 32);
      };
      auto load_q = [&](const Unit& U, int n, int t) {
        if (n > 0 && !(ok = wait_free(&ctl->q_empty[t], (n - 1) & 1, 16)))
          return;
        mbar_arrive_expect_tx(&ctl->q_full[t], C::kTileBytes);
        for (int x = 0; x < C::kBoxes; ++x)
          load_box(s_q + t * C::kTileBytes + x * (kBM * 128), &tm_q, &ctl->q_full[t],
                   x * C::kBoxCols, U.row_base + t * kBM, U.h, U.b, p.bshd);
      };
      auto load_kv = [&](const Unit& U, int j) {
#pragma unroll
        for (int kind = 0; kind < 2; ++kind) {
          const int st = issued % C::kStages;
          const int round = issued / C::kStages;
          if (round > 0 && !(ok = wait_free(&ctl->kv_empty[st], (round - 1) & 1, 10)))
            return;
          uint8_t* dst = s_kv + st * C::kTileBytes;
          mbar_arrive_expect_tx(&ctl->kv_full[st], C::kTileBytes);
          const CUtensorMap* map = kind == 0 ? &tm_k : &tm_v;
          for (int x = 0; x < C::kBoxes; ++x)
            load_box(dst + x * (kBN * 128), map, &ctl->kv_full[st], x * C::kBoxCols, j * kBN, U.h,
                     U.b, p.bshd);
          ++issued;
        }
      };
      // A unit is taken only when the previous one is fully issued, so
      // faster CTAs take more of the (unequal, causal) units.
      // Causal units have unequal lengths.  Head-major order (unit_info)
      // keeps the units in flight on a few heads, whose K/V stay in L2, but
      // the last heads' long units would start late and leave the other CTAs
      // idle at the end; so the last ~2 waves' worth of heads (their K/V
      // still fit in L2) hand out their units longest first across heads.
      // The producer maps the n-th unit taken to its head-major index once;
      // every role then decodes that index with unit_info.
      const int nbh = p.B * p.H;
      const int tail_bh = p.causal ? min(nbh, (2 * p.ctas + nqb - 1) / nqb) : 0;
      const int u_tail = (nbh - tail_bh) * nqb;
      auto head_major = [&](int u) {
        if (u < u_tail) return u;
        const int v = u - u_tail;
        return (nbh - tail_bh + v % tail_bh) * nqb + v / tail_bh;
      };
      for (int n = 0; ok; ++n) {
        int u = dyn ? atomicAdd(p.sched, 1) : (n == 0 ? static_cast<int>(blockIdx.x) : n_units);
        u = (u >= n_units || *abort_flag) ? -1 : head_major(u);
        const int slot = n & 1;
        if (n >= 2 && !(ok = wait_free(&ctl->unit_empty[slot], ((n >> 1) - 1) & 1, 17)))
          break;
        ctl->unit_ring[slot] = u;
        mbar_arrive(&ctl->unit_full[slot]);  // release: the id is visible to the waiters
        if (u < 0) break;
        const Unit U = unit_info(u);
        for (int j = 0; j < min(U.n_all, kL2PrefetchTiles); ++j)
          for (int x = 0; x < C::kBoxes; ++x) {
            prefetch_box(&tm_k, x * C::kBoxCols, j * kBN, U.h, U.b, p.bshd);
            prefetch_box(&tm_v, x * C::kBoxCols, j * kBN, U.h, U.b, p.bshd);
          }
        // Q_0, the first K/V tile, then Q_1: each Q tile is refilled as soon
        // as the previous unit's last S MMA of that tile has read it, and the
        // first K/V tile does not wait for the later Q tile.
        load_q(U, n, 0);
        if (ok && U.n_all > 0) load_kv(U, 0);
        if (ok) load_q(U, n, 1);
        if (!ok) break;
        q_loads = n + 1;
        for (int j = 1; j < U.n_all && ok && !*abort_flag; ++j) {
          if (j - 1 + kL2PrefetchTiles < U.n_all)
            for (int x = 0; x < C::kBoxes; ++x) {
              prefetch_box(&tm_k, x * C::kBoxCols, (j - 1 + kL2PrefetchTiles) * kBN, U.h, U.b,
                           p.bshd);
              prefetch_box(&tm_v, x * C::kBoxCols, (j - 1 + kL2PrefetchTiles) * kBN, U.h, U.b,
                           p.bshd);
            }
          load_kv(U, j);
        }
      }
      if (!ok) *abort_flag = 1;
      // Never leave the CTA with a copy still landing in shared memory: wait
      // (bounded) for the last load issued into every stage and for Q.
      for (int idx = max(0, issued - C::kStages); idx < issued; ++idx)
        mbar_wait(&ctl->kv_full[idx % C::kStages], (idx / C::kStages) & 1, p.wait_limit_ns,
                  p.err, 11);
      if (q_loads > 0)
        for (int t = 0; t < kTiles; ++t)
          mbar_wait(&ctl->q_full[t], (q_loads - 1) & 1, p.wait_limit_ns, p.err, 12);
    }
    __syncwarp();
   } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s =
          kFp8 ? idesc_e4m3(kBM, kBN, false, false) : idesc_f16(kBF16, kBM, kBN, false, false);
      constexpr uint32_t id_o =
          kFp8 ? idesc_e4m3(kBM, D, false, true) : idesc_f16(kBF16, kBM, D, false, true);
      const uint32_t q_addr = smem_u32(s_q);
      const uint32_t kv_addr = smem_u32(s_kv);
      bool ok = true;

      // Descriptors are built once; inside the loops each MMA only adds a
      // compile-time offset to a low word, so the issuing thread can feed
      // the tensor core's short instruction queue without a dependent chain
      // of address arithmetic.
      const uint32_t hi_k = sdesc_hi_sw128(1024);  // K-major: 8-row groups 1024 B apart
      const uint32_t q_lo = sdesc_lo(q_addr, 16);
      const uint32_t k_lo = sdesc_lo(kv_addr, 16);         // K-major: leading offset unused
      // V: 128-byte column groups 16 KB apart (FP8, D = 128: a single group)
      const uint32_t v_lo = sdesc_lo(kv_addr, kBN * 128);
      constexpr uint32_t kTileLo = C::kTileBytes >> 4;
      // S_t = Q_t K_j^T  (both operands K-major, 128-byte swizzle)
      auto issue_s = [&](int t, int st) {
        const uint32_t qa = q_lo + t * kTileLo;
        const uint32_t ka = k_lo + st * kTileLo;
        const uint32_t d = tmem + C::col_s(t);
#pragma unroll
        for (int kk = 0; kk < D * C::kElt / 32; ++kk) {  // 32 bytes of K per instruction
          const uint32_t off = ((kk / 4) * (kBM * 128) + (kk % 4) * 32) >> 4;
          mma_ss_lh<kFp8>(d, qa + off, hi_k, ka + off, hi_k, id_s, kk > 0);
        }
      };
      // O_t (+)= P_t V_j  (P from tensor memory, V MN-major, 128-byte swizzle)
      // Half `hf` covers keys [64*hf, 64*hf + 64); every instruction reads 8
      // tensor-memory columns of P (16 keys as 16-bit pairs, 32 as E4M3 quads).
      auto issue_pv_half = [&](int t, int st, bool acc, int hf) {
        const uint32_t va = v_lo + st * kTileLo;
        const uint32_t d = tmem + C::col_o(t);
        const uint32_t a = tmem + C::col_s(t);
        constexpr int kPerHalf = 64 / C::kKeysPerPV;
#pragma unroll
        for (int k4 = 0; k4 < kPerHalf; ++k4) {
          const int kk = hf * kPerHalf + k4;
          mma_ts_lh<kFp8>(d, a + kk * 8, va + ((kk * C::kKeysPerPV * 128) >> 4), hi_k, id_o,
                          (acc || kk > 0) ? 1u : 0u);
        }
      };
      // A K/V stage is free once this CTA's MMAs (and the partner's) read it.
      auto release = [&](int st) {
        if (cs == 2)
          mma_commit_multicast(&ctl->kv_empty[st], 0x3);
        else
          mma_commit(&ctl->kv_empty[st]);
      };
      auto wait_full = [&](int idx, int site) {
        return mbar_wait(&ctl->kv_full[idx % C::kStages], (idx / C::kStages) & 1,
                         p.wait_limit_ns, p.err, site);
      };

      int base = 0;         // K/V stages consumed by earlier units
      int np[kTiles] = {};  // P tiles consumed per query tile, all units
      for (int n = 0; ok; ++n) {
        if (!(ok = mbar_wait(&ctl->unit_full[n & 1], (n >> 1) & 1, p.wait_limit_ns, p.err, 28)))
          break;
        const int u = read_unit(n);
        mbar_arrive(&ctl->unit_empty[n & 1]);
        if (u < 0) break;
        const Unit U = unit_info(u);
        // Each query tile releases its Q (q_empty) after its last S MMA,
        // exactly once per unit, and signals its O (o_full) after its last PV
        // MMA, once per unit in which it has keys.  (A unit without keys
        // signalling o_full at once could complete two phases before a
        // waiter still on the previous unit looked, which it would then
        // never see.)
        if (U.n_all > 0 && !(ok = wait_full(base, 21))) break;
        for (int t = 0; t < kTiles && ok; ++t) {
          if (!(ok = mbar_wait(&ctl->q_full[t], n & 1, p.wait_limit_ns, p.err, 20))) break;
          tc_fence_after_sync();
          if (U.n_kv(t) > 0) {
            issue_s(t, base % C::kStages);
            mma_commit(&ctl->s_full[t]);
          }
          if (U.n_kv(t) <= 1) mma_commit(&ctl->q_empty[t]);
        }
        if (!ok) break;
        if (U.n_all > 0) release(base % C::kStages);
        for (int j = 0; j < U.n_all && ok; ++j) {
          const int st_v = (base + 2 * j + 1) % C::kStages;
          const int st_kn = (base + 2 * j + 2) % C::kStages;
          const bool next = j + 1 < U.n_all;
          bool kn_ready = false;
          if (!(ok = wait_full(base + 2 * j + 1, 22))) break;
          for (int t = 0; t < kTiles && ok; ++t) {
            if (j < U.n_kv(t)) {
              // The first PV of a unit overwrites O_t: the previous unit's
              // epilogue must hold it in registers by then.
              if (j == 0 && n > 0 &&
                  !(ok = mbar_wait(&ctl->o_free[t], (n - 1) & 1, p.wait_limit_ns, p.err, 29)))
                break;
              // One wait per P tile, then all of P_t V_j as one batch: each
              // wait of this thread costs the tensor core idle time once the
              // queue behind it has drained, and publishing P in two halves
              // (PV of keys 0-63 started early) measured 2-5% slower.
              if (!(ok = mbar_wait(&ctl->p_full[t], np[t] & 1, p.wait_limit_ns, p.err, 23 + t)))
                break;
              tc_fence_after_sync();
              issue_pv_half(t, st_v, j > 0, 0);
              issue_pv_half(t, st_v, j > 0, 1);
              ++np[t];
              if (j == U.n_kv(t) - 1) mma_commit(&ctl->o_full[t]);
            }
            if (t == kTiles - 1) release(st_v);
            if (next) {
              if (!kn_ready) {
                if (!(ok = wait_full(base + 2 * j + 2, 25))) break;
                kn_ready = true;
                tc_fence_after_sync();
              }
              if (j + 1 < U.n_kv(t)) {
                issue_s(t, st_kn);
                mma_commit(&ctl->s_full[t]);
                if (j + 1 == U.n_kv(t) - 1) mma_commit(&ctl->q_empty[t]);
              }
              if (t == kTiles - 1) release(st_kn);
            }
          }
        }
        base += 2 * U.n_all;
      }
      if (!ok) *abort_flag = 1;
    }
    __syncwarp();
    // Release tensor memory once every softmax warp has read its last O
    // (which follows every MMA of this CTA).
    mbar_wait(&ctl->tmem_free, 0, p.wait_limit_ns, p.err, 27);
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
   }
  } else {
    // ============================================= softmax warpgroups
    setmaxnreg_inc<kRegsSoftmax>();
    const int t = warp / 4;             // query tile of this warpgroup
    const int wl = warp % 4;            // warp's TMEM lane quarter
    const int r = wl * 32 + lane;       // row within the tile
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wl * 32) << 16);
    const uint32_t col_s = C::col_s(t);
    const uint32_t col_o = C::col_o(t);
    const float c = p.scale_log2;
    int ns = 0;   // S tiles of this query tile consumed, all units
    int nof = 0;  // O tiles of this query tile with keys consumed, all units
    bool ok = true;
    for (int n = 0; ok; ++n) {
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->unit_full[n & 1], (n >> 1) & 1,
                                             p.wait_limit_ns, p.err, 42));
      if (!ok) break;
      const int u = read_unit(n);
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->unit_empty[n & 1]);
      if (u < 0) break;
      // Only what this tile needs of the unit stays live through the loop.
      int b, h, S_kv, row0, n_kv;
      {
        const Unit U = unit_info(u);
        b = U.b;
        h = U.h;
        S_kv = U.S_kv;
        row0 = U.row_base + t * kBM;
        n_kv = U.n_kv(t);
      }
      const int i = row0 + r;             // query index
      const int diag = S_kv - p.S_q;      // bottom-right causal offset

      float m2 = -INFINITY;  // running reference max, scaled log2 units
      float l = 0.f;         // running sum of exponentials relative to m2
      for (int j = 0; j < n_kv; ++j, ++ns) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&ctl->s_full[t], ns & 1, p.wait_limit_ns, p.err, 30 + t));
        if (!ok) break;
        tc_fence_after_sync();
        float s[kBN];
        tmem_ld128_wait(lane_addr + col_s, s);
        const int key0 = j * kBN;
        const bool full = (key0 + kBN <= S_kv) && (!p.causal || key0 + kBN - 1 <= row0 + diag);
        if (!full) {
          // Keys past L = lim - key0 (this row's last visible column of the
          // tile) are masked.  L never decreases with the row, so the warp's
          // first row bounds it below: a 32-column quarter every row of the
          // warp sees in full (a warp-uniform test) needs no compares.
          const int lim = p.causal ? min(S_kv - 1, i + diag) : S_kv - 1;
          const int L = lim - key0;
          const int row_w = row0 + wl * 32;  // the warp's first row
          const int l_lo = (p.causal ? min(S_kv - 1, row_w + diag) : S_kv - 1) - key0;
#pragma unroll
          for (int qq = 0; qq < kBN / 32; ++qq) {
            if (l_lo < 32 * qq + 31) {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (32 * qq + e > L) s[32 * qq + e] = -INFINITY;
            }
          }
        }
        // Row max: eight independent chains of 3-input max, then a short tree.
        float mx[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mx[q] = fmax3(s[3 * q], s[3 * q + 1], s[3 * q + 2]);  // 0..23
#pragma unroll
        for (int cc = 24; cc < kBN - 8; cc += 16)
#pragma unroll
          for (int q = 0; q < 8; ++q) mx[q] = fmax3(mx[q], s[cc + 2 * q], s[cc + 2 * q + 1]);
        // columns 24 .. 119 consumed; 120 .. 127 remain
#pragma unroll
        for (int q = 0; q < 8; ++q) mx[q] = fmaxf(mx[q], s[kBN - 8 + q]);
        const float m_raw = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                  fmaxf(mx[6], mx[7]));
        const float m_new = fmaxf(m2, m_raw * c);
        float alpha = 1.f;
        bool need = false;
        if (m_new > m2 + kRescaleThreshold) {  // false while m_new == -inf
          alpha = ex2_approx(m2 - m_new);      // 0 on the first visible tile
          need = (j > 0);
          m2 = m_new;
        }
        if (__any_sync(0xffffffffu, need)) {
          // O_t row *= alpha before any of P_t,j is published.  PV_t,j-1
          // completed before S_t,j was signalled.
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 32) {
            uint32_t o[32];
            tmem_ld32_wait(lane_addr + col_o + cc, o);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
            tmem_st32(lane_addr + col_o + cc, o);
          }
        }
        const float mref = (m2 == -INFINITY) ? 0.f : m2;
        const uint64_t c2 = f2_pack(c, c);
        const uint64_t nm2 = f2_pack(-mref, -mref);
        uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if constexpr (kFp8) {
            uint32_t pk[16];  // 64 keys as E4M3, four per column
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              float x0, x1, x2, x3;
              f2_unpack(f2_fma(f2_pack(s[half * 64 + 4 * q], s[half * 64 + 4 * q + 1]), c2, nm2),
                        x0, x1);
              f2_unpack(f2_fma(f2_pack(s[half * 64 + 4 * q + 2], s[half * 64 + 4 * q + 3]), c2,
                               nm2),
                        x2, x3);
              const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
              const float e2 = ex2_approx(x2), e3 = ex2_approx(x3);
              acc0 = f2_add(acc0, f2_pack(e0, e1));
              acc1 = f2_add(acc1, f2_pack(e2, e3));
              pk[q] = pack4_e4m3(e0, e1, e2, e3);
            }
            tmem_st16(lane_addr + col_s + half * 16, pk);
          } else {
            uint32_t pk[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(s[half * 64 + 2 * q], s[half * 64 + 2 * q + 1]), c2, nm2),
                        x0, x1);
              const float e0 = ex2_approx(x0);
              const float e1 = ex2_approx(x1);
              if (q & 1)
                acc1 = f2_add(acc1, f2_pack(e0, e1));
              else
                acc0 = f2_add(acc0, f2_pack(e0, e1));
              pk[q] = pack2<kBF16>(e0, e1);
            }
            tmem_st32(lane_addr + col_s + half * 32, pk);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full[t]);
        float a0, a1, b0, b1;
        f2_unpack(acc0, a0, a1);
        f2_unpack(acc1, b0, b1);
        l = l * alpha + ((a0 + a1) + (b0 + b1));
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      if (n_kv > 0) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&ctl->o_full[t], nof & 1, p.wait_limit_ns, p.err, 40 + t));
        if (!ok) break;
        ++nof;
        tc_fence_after_sync();
      }
      const bool have_o = n_kv > 0 && l > 0.f;
      const float inv_l = have_o ? p.o_scale / l : 0.f;
      if constexpr (kPaged) {
        // One unit per CTA: Q_t is dead and holds O_t for a TMA store.  With
        // keys, the last PV MMA (o_full) followed every read of Q_t; without,
        // only Q_t's own load may still be landing there.
        uint8_t* s_o = s_q + t * C::kTileBytes;
        if (n_kv == 0) {
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&ctl->q_full[t], 0, p.wait_limit_ns, p.err, 39));
          if (!ok) break;
        }
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 64) {
          uint32_t o[64] = {};
          if (n_kv > 0) tmem_ld64_wait(lane_addr + col_o + cc, o);
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
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->o_free[t]);
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
      } else {
        if constexpr (C::kStagedO) {
          // O_t is staged in this query tile's own shared-memory tile (Q_t
          // already holds the next unit) and leaves by TMA store.  The thread
          // that issues the store first waits until its previous store has
          // read the tile; the loads from tensor memory run meanwhile.
          uint8_t* s_o = smem + C::kOStageOff + t * C::kOTileBytes;
          const bool issuer = wl == 0 && lane == 0;
          uint32_t o[D];
#pragma unroll
          for (int cc = 0; cc < D; cc += 64) {
            if (n_kv > 0) {
              tmem_ld64_wait(lane_addr + col_o + cc, *reinterpret_cast<uint32_t(*)[64]>(o + cc));
            } else {
#pragma unroll
              for (int e = 0; e < 64; ++e) o[cc + e] = 0u;
            }
          }
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->o_free[t]);
          if (issuer) tma_store_wait_read_all();
          named_barrier_sync(1 + t, 128);
#pragma unroll
          for (int cc = 0; cc < D; cc += 64) {
            uint8_t* sub = s_o + (cc / 64) * (kBM * 128) + r * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) {  // 8 chunks of 8 columns = 16 bytes each
              uint4 w;
              uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float v0 = have_o ? __uint_as_float(o[cc + q * 8 + 2 * e]) * inv_l : 0.f;
                const float v1 =
                    have_o ? __uint_as_float(o[cc + q * 8 + 2 * e + 1]) * inv_l : 0.f;
                wp[e] = pack2<kBF16>(v0, v1);
              }
              *reinterpret_cast<uint4*>(sub + ((q ^ (r & 7)) * 16)) = w;
            }
          }
          fence_proxy_async_smem();
          named_barrier_sync(1 + t, 128);
          if (issuer && row0 < p.S_q) {
            for (int x = 0; x < D / 64; ++x)
              if (p.bshd)
                tma_store_4d(&tm_o, s_o + x * (kBM * 128), x * 64, h, row0, b);
              else
                tma_store_4d(&tm_o, s_o + x * (kBM * 128), x * 64, row0, h, b);
            tma_store_commit();
          }
          __syncwarp();
        } else {
          // Q_t already holds the next unit's rows: O_t goes from registers
          // straight to global memory, one 16-byte store per 8 columns of the
          // thread's row, after the registers release tensor memory.
          uint32_t o[D];
#pragma unroll
          for (int cc = 0; cc < D; cc += 64) {
            if (n_kv > 0) {
              tmem_ld64_wait(lane_addr + col_o + cc, *reinterpret_cast<uint32_t(*)[64]>(o + cc));
            } else {
#pragma unroll
              for (int e = 0; e < 64; ++e) o[cc + e] = 0u;
            }
          }
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->o_free[t]);
          if (i < p.S_q) {
            // A row is D 16-bit values (128 or 256 bytes, 32-byte aligned):
            // whole 32-byte sectors, one store each.
            const size_t row = p.bshd ? (static_cast<size_t>(b) * p.S_q + i) * p.H + h
                                      : (static_cast<size_t>(b) * p.H + h) * p.S_q + i;
            uint16_t* dst = static_cast<uint16_t*>(p.o) + row * D;
#pragma unroll
            for (int q = 0; q < D / 16; ++q) {
              uint32_t w[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float v0 = have_o ? __uint_as_float(o[q * 16 + 2 * e]) * inv_l : 0.f;
                const float v1 = have_o ? __uint_as_float(o[q * 16 + 2 * e + 1]) * inv_l : 0.f;
                w[e] = pack2<kBF16>(v0, v1);
              }
              if (p.o_align32) {  // the base is 32-byte aligned (checked on the host)
                st_global_v8(dst + q * 16, w);
              } else {
                uint4* d4 = reinterpret_cast<uint4*>(dst + q * 16);
                d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
                d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
              }
            }
          }
        }
      }
      if (p.lse != nullptr && i < p.S_q) {
        const float lse = have_o ? (m2 + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        p.lse[(static_cast<size_t>(b) * p.H + h) * p.S_q + i] = lse;
      }
    }
    // No O store may still be reading shared memory when the CTA exits.
    if (C::kStagedO && wl == 0 && lane == 0) tma_store_wait_all();
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->tmem_free);
  }
  // Stay resident until the partner has made its last multicast and commit.
  if (cs == 2) cluster_sync();
}

}  // namespace

template <int D, bool kBF16, bool kPaged, bool kFp8 = false>
static cudaError_t launch_one(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                              const CUtensorMap& o, const PrefillParams& p, int grid,
                              cudaStream_t stream) {
  auto kern = prefill_fwd_kernel<D, kBF16, kPaged, kFp8>;
  static std::atomic<unsigned long long> configured{0};  // per template instance, per device
  cudaError_t ce = attn_host::once_per_device(configured, [&]() {
    // The in-kernel register split assumes exactly kRegsAtLaunch registers
    // per thread at launch; with fewer, setmaxnreg.inc would never complete.
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kRegsAtLaunch) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<D, kFp8, kPaged>::kSmemBytes);
  });
  if (ce != cudaSuccess) return ce;
  if (!(kPaged && p.pair)) {
    kern<<<grid, kThreads, Cfg<D, kFp8, kPaged>::kSmemBytes, stream>>>(q, k, v, o, p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<D, kFp8, kPaged>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, q, k, v, o, p);
}

// Persistent CTAs (one per SM) when the host passes a zeroed scheduler
// counter, else one CTA per unit.
static int contiguous_grid(const PrefillParams& p) {
  const int units = p.B * p.H * p.num_q_blocks;
  return (p.sched != nullptr && p.ctas > 0 && p.ctas < units) ? p.ctas : units;
}

cudaError_t prefill_launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const CUtensorMap& o, const PrefillParams& p, int D, bool bf16,
                           cudaStream_t stream) {
  const int grid = contiguous_grid(p);
  if (grid == 0) return cudaSuccess;
  if (D == 128) return bf16 ? launch_one<128, true, false>(q, k, v, o, p, grid, stream)
                            : launch_one<128, false, false>(q, k, v, o, p, grid, stream);
  return bf16 ? launch_one<64, true, false>(q, k, v, o, p, grid, stream)
              : launch_one<64, false, false>(q, k, v, o, p, grid, stream);
}

cudaError_t extend_launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& o, const PrefillParams& p, int D, bool bf16,
                          cudaStream_t stream) {
  const int grid = p.B * p.H * p.num_q_blocks;
  if (grid == 0) return cudaSuccess;
  if (D == 128) return bf16 ? launch_one<128, true, true>(q, k, v, o, p, grid, stream)
                            : launch_one<128, false, true>(q, k, v, o, p, grid, stream);
  return bf16 ? launch_one<64, true, true>(q, k, v, o, p, grid, stream)
              : launch_one<64, false, true>(q, k, v, o, p, grid, stream);
}

cudaError_t prefill_fp8_launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& o, const PrefillParams& p, bool bf16_out,
                               cudaStream_t stream) {
  const int grid = contiguous_grid(p);
  if (grid == 0) return cudaSuccess;
  return bf16_out ? launch_one<128, true, false, true>(q, k, v, o, p, grid, stream)
                  : launch_one<128, false, false, true>(q, k, v, o, p, grid, stream);
}

int prefill_rows_per_cta() { return kTiles * kBM; }
int prefill_box_rows() { return kBM; }

}  // namespace attn_sm103a
