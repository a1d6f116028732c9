// attn_api.cu -- the C ABI (include/attn_gb300.h): argument validation, TMA
// tensor-map encoding, the decode split plan and workspace, error reporting.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/attn_gb300.h"
#include "backward_sm103a.h"
#include "decode_plan.h"
#include "decode_sm103a.h"
#include "mqa_logits_sm103a.h"
#include "prefill_sm103a.h"
#include "sm103a_ptx.cuh"
#include "tmap.h"

namespace {

constexpr uint64_t kDefaultWaitLimitNs = 4000000000ull;  // 4 s
constexpr int kMaxDevices = 64;

thread_local std::string t_last_error;

uint64_t initial_wait_limit() {
  const char* v = std::getenv("ATTN_WAIT_LIMIT_NS");
  if (v && *v) {
    unsigned long long n = std::strtoull(v, nullptr, 10);
    if (n > 0) return n;
  }
  return kDefaultWaitLimitNs;
}

std::atomic<uint64_t> g_wait_limit_ns{initial_wait_limit()};

__device__ int g_device_error_word = 0;

attn_status fail(attn_status s, const std::string& msg) {
  t_last_error = msg;
  return s;
}

attn_status fail_cuda(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

struct DeviceState {
  std::mutex mu;
  int* err_word = nullptr;    // device address of g_device_error_word
  int num_sms = 0;
  // Decode split partials, one buffer per stream: calls on different streams
  // may overlap on the GPU, calls on one stream run in order.
  struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
  };
  std::unordered_map<cudaStream_t, Workspace> workspaces;
  // Buffers a workspace outgrew: still referenced by any graph captured while
  // they were current, so kept until attn_release_workspace.
  std::vector<void*> retired;
  // Prefill unit counters (one int per stream): persistent CTAs take their
  // next query block from it; the host zeroes it before every launch.
  std::unordered_map<cudaStream_t, int*> sched;
};

// The stream's prefill unit counter, created on first use outside stream
// capture.  nullptr (one CTA per unit instead) while a stream without one is
// being captured.
attn_status prefill_sched(DeviceState* st, cudaStream_t stream, int** out) {
  *out = nullptr;
  std::lock_guard<std::mutex> lk(st->mu);
  auto it = st->sched.find(stream);
  if (it == st->sched.end()) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone) return ATTN_OK;
    int* c = nullptr;
    e = cudaMalloc(&c, 16);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(ATTN_ERR_NO_MEMORY, std::string("scheduler cudaMalloc: ") + cudaGetErrorString(e));
    }
    it = st->sched.emplace(stream, c).first;
  }
  cudaError_t e = cudaMemsetAsync(it->second, 0, sizeof(int), stream);
  if (e != cudaSuccess) return fail_cuda(e, "scheduler reset");
  *out = it->second;
  return ATTN_OK;
}

DeviceState g_dev[kMaxDevices];

// A wait that nothing completes: one thread initialises an mbarrier nobody
// arrives on and waits for its first phase with the kernels' bounded wait,
// which gives up after limit_ns and records (timeout << 16) | kSelftestSite
// in the error word.  No copy, MMA or tensor memory is involved.
constexpr int kSelftestSite = 900;
__global__ void selftest_wait_kernel(int* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  attn_sm103a::mbar_init(&bar, 1);
  attn_sm103a::fence_mbar_init();
  attn_sm103a::mbar_wait(&bar, 0, limit_ns, err, kSelftestSite);
}

// Per-device set-up, done once with the device current.
attn_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device index too large");
  DeviceState& st = g_dev[dev];
  std::lock_guard<std::mutex> lk(st.mu);
  if (st.err_word == nullptr) {
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err_word), g_device_error_word);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(error word)");
    e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute(SM count)");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) {
      st.err_word = nullptr;
      return fail(ATTN_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300) only; device is sm_" +
                                            std::to_string(major) + std::to_string(minor));
    }
  }
  *out = &st;
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Prefill tensor map over a [B,H,S,D] (BHSD) or [B,S,H,D] (BSHD) tensor.
// BHSD dims (D, S, H, B); BSHD dims (D, H, S, B) so strides grow outward.
bool prefill_map(CUtensorMap* m, const void* base, int B, int H, int S, int D, bool bshd,
                 bool bf16) {
  const uint64_t el = 2;
  uint64_t dims[4], strides[3];
  uint32_t box[4];
  if (!bshd) {
    dims[0] = D; dims[1] = S; dims[2] = H; dims[3] = B;
    strides[0] = el * D; strides[1] = el * D * S; strides[2] = el * D * S * H;
    box[0] = 64; box[1] = attn_sm103a::prefill_box_rows(); box[2] = 1; box[3] = 1;
  } else {
    dims[0] = D; dims[1] = H; dims[2] = S; dims[3] = B;
    strides[0] = el * D; strides[1] = el * D * H; strides[2] = el * D * H * S;
    box[0] = 64; box[1] = 1; box[2] = attn_sm103a::prefill_box_rows(); box[3] = 1;
  }
  return attn_host::encode_tiled_16bit(m, base, 4, dims, strides, box, bf16,
                                       CU_TENSOR_MAP_SWIZZLE_128B);
}

// FP8 prefill tensor map over E4M3 bytes, layouts as prefill_map; box 128
// columns (128 bytes) x 128 rows.
bool prefill_map_fp8(CUtensorMap* m, const void* base, int B, int H, int S, int D, bool bshd) {
  uint64_t dims[4], strides[3];
  uint32_t box[4];
  if (!bshd) {
    dims[0] = D; dims[1] = S; dims[2] = H; dims[3] = B;
    strides[0] = D; strides[1] = static_cast<uint64_t>(D) * S;
    strides[2] = static_cast<uint64_t>(D) * S * H;
    box[0] = 128; box[1] = attn_sm103a::prefill_box_rows(); box[2] = 1; box[3] = 1;
  } else {
    dims[0] = D; dims[1] = H; dims[2] = S; dims[3] = B;
    strides[0] = D; strides[1] = static_cast<uint64_t>(D) * H;
    strides[2] = static_cast<uint64_t>(D) * H * S;
    box[0] = 128; box[1] = 1; box[2] = attn_sm103a::prefill_box_rows(); box[3] = 1;
  }
  return attn_host::encode_tiled_8bit(m, base, 4, dims, strides, box,
                                      CU_TENSOR_MAP_SWIZZLE_128B);
}

// Decode tensor map over a pool [num_pages, page_size, H_kv, D]: dims
// (D, H_kv, page_size, num_pages), box (64, 1, rows, 1).
bool decode_map(CUtensorMap* m, const void* base, int num_pages, int page_size, int H_kv, int D,
                int box_rows, bool bf16) {
  const uint64_t el = 2;
  uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(H_kv),
                      static_cast<uint64_t>(page_size), static_cast<uint64_t>(num_pages)};
  uint64_t strides[3] = {el * D, el * D * H_kv, el * D * H_kv * page_size};
  uint32_t box[4] = {64, 1, static_cast<uint32_t>(box_rows), 1};
  return attn_host::encode_tiled_16bit(m, base, 4, dims, strides, box, bf16,
                                       CU_TENSOR_MAP_SWIZZLE_128B,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// Extend tensor map over a pool [num_pages, page_size, H_kv, D] seen as 2-D:
// dims (H_kv * D, num_pages * page_size), box (64, rows).
bool extend_map(CUtensorMap* m, const void* base, int num_pages, int page_size, int H_kv, int D,
                int box_rows, bool bf16) {
  const uint64_t el = 2;
  uint64_t dims[2] = {static_cast<uint64_t>(D) * H_kv,
                      static_cast<uint64_t>(num_pages) * page_size};
  uint64_t strides[1] = {el * D * H_kv};
  uint32_t box[2] = {64, static_cast<uint32_t>(box_rows)};
  return attn_host::encode_tiled_16bit(m, base, 2, dims, strides, box, bf16,
                                       CU_TENSOR_MAP_SWIZZLE_128B,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  return std::atoi(v);
}

}  // namespace

extern "C" {

const char* attn_version(void) { return "attn_gb300 0.1.0 (sm_103a)"; }

const char* attn_last_error(void) { return t_last_error.c_str(); }

void attn_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns ? ns : initial_wait_limit());
}

attn_status attn_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull)
    return fail(ATTN_ERR_INVALID_ARG, "limit_ns must be in (0, 1e10]");
  DeviceState* st = nullptr;
  attn_status s = device_state(&st);
  if (s != ATTN_OK) return s;
  selftest_wait_kernel<<<1, 1, 0, stream>>>(st->err_word, limit_ns);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "self-test launch");
  return ATTN_OK;
}

attn_status attn_device_error(int* word, int clear) {
  DeviceState* st = nullptr;
  attn_status s = device_state(&st);
  if (s != ATTN_OK) return s;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize");
  int w = 0;
  e = cudaMemcpy(&w, st->err_word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e, "read device error word");
  if (clear && w != 0) {
    int zero = 0;
    e = cudaMemcpy(st->err_word, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_cuda(e, "clear device error word");
  }
  if (word) *word = w;
  if (w != 0) {
    char buf[96];
    std::snprintf(buf, sizeof(buf), "device error word 0x%08x (code %d, site %d)", w, w >> 16,
                  w & 0xFFFF);
    return fail(ATTN_ERR_DEVICE_TIMEOUT, buf);
  }
  return ATTN_OK;
}

attn_status attn_prefill_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int S_q, int S_kv, int D, attn_layout layout,
                             attn_dtype dtype, int causal, float scale, cudaStream_t stream) {
  if (B < 0 || H < 0 || S_q < 0 || S_kv < 0)
    return fail(ATTN_ERR_INVALID_ARG, "B, H, S_q and S_kv must be >= 0");
  if (layout != ATTN_BHSD && layout != ATTN_BSHD)
    return fail(ATTN_ERR_INVALID_ARG, "layout must be ATTN_BHSD or ATTN_BSHD");
  if (dtype != ATTN_F16 && dtype != ATTN_BF16)
    return fail(ATTN_ERR_INVALID_ARG, "dtype must be ATTN_F16 or ATTN_BF16");
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!(std::isfinite(scale) && scale > 0.f))
    return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (D != 64 && D != 128) return fail(ATTN_ERR_UNSUPPORTED, "D must be 64 or 128");
  if (static_cast<int64_t>(B) * H * S_q == 0) return ATTN_OK;  // nothing to compute
  if (!q || !o || (S_kv > 0 && (!k || !v)))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be non-NULL");
  if (!aligned16(q) || !aligned16(o) || (S_kv > 0 && (!aligned16(k) || !aligned16(v))))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  const int64_t elems = static_cast<int64_t>(B) * H * (S_q > S_kv ? S_q : S_kv) * D;
  if (elems * 2 >= (int64_t(1) << 40))
    return fail(ATTN_ERR_UNSUPPORTED, "tensor too large for one TMA descriptor");
  const int rows = attn_sm103a::prefill_rows_per_cta();
  const int64_t n_qb = (S_q + rows - 1) / rows;
  if (static_cast<int64_t>(B) * H * n_qb > 0x7FFFFFFF)
    return fail(ATTN_ERR_UNSUPPORTED, "grid too large");

  DeviceState* st = nullptr;
  attn_status s = device_state(&st);
  if (s != ATTN_OK) return s;

  const bool bshd = layout == ATTN_BSHD;
  const bool bf16 = dtype == ATTN_BF16;
  CUtensorMap mq, mk, mv, mo;
  // With S_kv == 0 no K/V tile is ever loaded; q stands in as a valid base.
  const int S_kv_map = S_kv > 0 ? S_kv : 1;
  const void* kb = S_kv > 0 ? k : q;
  const void* vb = S_kv > 0 ? v : q;
  if (!prefill_map(&mq, q, B, H, S_q, D, bshd, bf16) ||
      !prefill_map(&mk, kb, B, H, S_kv_map, D, bshd, bf16) ||
      !prefill_map(&mv, vb, B, H, S_kv_map, D, bshd, bf16) ||
      !prefill_map(&mo, o, B, H, S_q, D, bshd, bf16))
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for a prefill tensor");

  attn_sm103a::PrefillParams p{};
  p.lse = lse;
  p.o_scale = 1.f;
  p.B = B;
  p.H = H;
  p.S_q = S_q;
  p.S_kv = S_kv;
  p.num_q_blocks = static_cast<int>(n_qb);
  p.causal = causal;
  p.bshd = bshd ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = st->err_word;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.o = o;
  p.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0 ? 1 : 0;
  p.ctas = st->num_sms;
  s = prefill_sched(st, stream, &p.sched);
  if (s != ATTN_OK) return s;
  cudaError_t e = attn_sm103a::prefill_launch(mq, mk, mv, mo, p, D, bf16, stream);
  if (e != cudaSuccess) return fail_cuda(e, "prefill launch");
  return ATTN_OK;
}

attn_status attn_mqa_logits_fp8(const void* q, const void* kv, const float* kv_scale,
                                const float* weights, const int32_t* window_start,
                                const int32_t* window_end, float* logits, int S_q, int S_kv,
                                int H, int D, int64_t logits_stride, int clean_logits,
                                cudaStream_t stream) {
  if (S_q < 0 || S_kv < 0) return fail(ATTN_ERR_INVALID_ARG, "S_q and S_kv must be >= 0");
  if (H != 32 && H != 64 && H != 128)
    return fail(ATTN_ERR_UNSUPPORTED, "H must be 32, 64 or 128");
  if (D != 128) return fail(ATTN_ERR_UNSUPPORTED, "D must be 128");
  if (clean_logits != 0 && clean_logits != 1)
    return fail(ATTN_ERR_INVALID_ARG, "clean_logits must be 0 or 1");
  if (logits_stride < S_kv) return fail(ATTN_ERR_INVALID_ARG, "logits_stride must be >= S_kv");
  if (static_cast<int64_t>(S_q) * S_kv == 0) return ATTN_OK;
  if (!q || !kv || !kv_scale || !weights || !window_start || !window_end || !logits)
    return fail(ATTN_ERR_INVALID_ARG, "every pointer must be non-NULL");
  if (!aligned16(q) || !aligned16(kv))
    return fail(ATTN_ERR_INVALID_ARG, "q and kv must be 16-byte aligned");
  if ((static_cast<int64_t>(S_q) + attn_sm103a::mqa_rows_per_block(H)) * H > 0x7FFFFFFF ||
      S_kv > 0x7FFFFF00)
    return fail(ATTN_ERR_UNSUPPORTED, "too many rows for one TMA descriptor");

  DeviceState* st = nullptr;
  attn_status s = device_state(&st);
  if (s != ATTN_OK) return s;

  CUtensorMap mq, mk;
  {
    uint64_t dims[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(S_q) * H};
    uint64_t strides[1] = {static_cast<uint64_t>(D)};
    uint32_t box[2] = {128, static_cast<uint32_t>(attn_sm103a::mqa_rows_per_slab_box())};
    if (!attn_host::encode_tiled_8bit(&mq, q, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for q");
  }
  {
    uint64_t dims[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(S_kv)};
    uint64_t strides[1] = {static_cast<uint64_t>(D)};
    uint32_t box[2] = {128, static_cast<uint32_t>(attn_sm103a::mqa_keys_per_tile())};
    if (!attn_host::encode_tiled_8bit(&mk, kv, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for kv");
  }
  attn_sm103a::MqaParams p{};
  p.kv_scale = kv_scale;
  p.w = weights;
  p.start = window_start;
  p.end = window_end;
  p.logits = logits;
  p.stride = logits_stride;
  p.S_q = S_q;
  p.S_kv = S_kv;
  p.H = H;
  p.clean = clean_logits;
  p.tiles_per_cta = attn_sm103a::mqa_tiles_per_cta(S_q, S_kv, H, st->num_sms);
  p.err = st->err_word;
  p.wait_limit_ns = g_wait_limit_ns.load();
  cudaError_t e = attn_sm103a::mqa_logits_launch(mq, mk, p, stream);
  if (e != cudaSuccess) return fail_cuda(e, "MQA logits launch");
  return ATTN_OK;
}

attn_status attn_prefill_bwd(const void* q, const void* k, const void* v, const void* o,
                             const void* dout, const float* lse, void* dq, void* dk, void* dv,
                             float* delta, int B, int H, int S_q, int S_kv, int D,
                             attn_layout layout, attn_dtype dtype, int causal, float scale,
                             cudaStream_t stream) {
  if (B < 0 || H < 0 || S_q < 0 || S_kv < 0)
    return fail(ATTN_ERR_INVALID_ARG, "B, H, S_q and S_kv must be >= 0");
  if (layout != ATTN_BHSD && layout != ATTN_BSHD)
    return fail(ATTN_ERR_INVALID_ARG, "layout must be ATTN_BHSD or ATTN_BSHD");
  if (dtype != ATTN_F16 && dtype != ATTN_BF16)
    return fail(ATTN_ERR_INVALID_ARG, "dtype must be ATTN_F16 or ATTN_BF16");
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!(std::isfinite(scale) && scale > 0.f))
    return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (D != 128) return fail(ATTN_ERR_UNSUPPORTED, "the backward supports D = 128 only");
  if (static_cast<int64_t>(B) * H == 0 || (S_q == 0 && S_kv == 0)) return ATTN_OK;
  if (S_q == 0 || S_kv == 0)
    return fail(ATTN_ERR_UNSUPPORTED, "the backward needs S_q > 0 and S_kv > 0");
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !delta)
    return fail(ATTN_ERR_INVALID_ARG, "every tensor pointer must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v, o, dout, dq, dk and dv must be 16-byte aligned");
  const int64_t elems = static_cast<int64_t>(B) * H * (S_q > S_kv ? S_q : S_kv) * D;
  if (elems * 2 >= (int64_t(1) << 40))
    return fail(ATTN_ERR_UNSUPPORTED, "tensor too large for one TMA descriptor");
  const int64_t tiles = static_cast<int64_t>(B) * H * ((S_q > S_kv ? S_q : S_kv) + 127) / 128;
  if (tiles > 0x7FFFFFFF || static_cast<int64_t>(B) * H * S_q / 8 > 0x7FFFFFFF)
    return fail(ATTN_ERR_UNSUPPORTED, "grid too large");

  DeviceState* st = nullptr;
  attn_status s = device_state(&st);
  if (s != ATTN_OK) return s;

  const bool bshd = layout == ATTN_BSHD;
  const bool bf16 = dtype == ATTN_BF16;
  CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
  if (!prefill_map(&mq, q, B, H, S_q, D, bshd, bf16) ||
      !prefill_map(&mk, k, B, H, S_kv, D, bshd, bf16) ||
      !prefill_map(&mv, v, B, H, S_kv, D, bshd, bf16) ||
      !prefill_map(&mdo, dout, B, H, S_q, D, bshd, bf16) ||
      !prefill_map(&mdq, dq, B, H, S_q, D, bshd, bf16) ||
      !prefill_map(&mdk, dk, B, H, S_kv, D, bshd, bf16) ||
      !prefill_map(&mdv, dv, B, H, S_kv, D, bshd, bf16))
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for a backward tensor");

  attn_sm103a::BackwardParams p{};
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.delta = delta;
  p.B = B;
  p.H = H;
  p.S_q = S_q;
  p.S_kv = S_kv;
  p.causal = causal;
  p.bshd = bshd ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = st->err_word;
  p.wait_limit_ns = g_wait_limit_ns.load();
  cudaError_t e = attn_sm103a::backward_launch(mq, mk, mv, mdo, mdq, mdk, mdv, p, bf16, stream);
  if (e != cudaSuccess) return fail_cuda(e, "backward launch");
  return ATTN_OK;
}

attn_status attn_prefill_fp8_fwd(const void* q, const void* k, const void* v, void* o,
                                 float* lse, int B, int H, int S_q, int S_kv, int D,
                                 attn_layout layout, attn_dtype out_dtype, int causal, float scale,
                                 float descale_q, float descale_k, float descale_v,
                                 cudaStream_t stream) {
  if (B < 0 || H < 0 || S_q < 0 || S_kv < 0)
    return fail(ATTN_ERR_INVALID_ARG, "B, H, S_q and S_kv must be >= 0");
  if (layout != ATTN_BHSD && layout != ATTN_BSHD)
    return fail(ATTN_ERR_INVALID_ARG, "layout must be ATTN_BHSD or ATTN_BSHD");
  if (out_dtype != ATTN_F16 && out_dtype != ATTN_BF16)
    return fail(ATTN_ERR_INVALID_ARG, "out_dtype must be ATTN_F16 or ATTN_BF16");
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!(std::isfinite(scale) && scale > 0.f))
    return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (!(std::isfinite(descale_q) && descale_q > 0.f && std::isfinite(descale_k) &&
        descale_k > 0.f && std::isfinite(descale_v) && descale_v > 0.f))
    return fail(ATTN_ERR_INVALID_ARG, "descale factors must be finite and > 0");
  if (D != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 form supports D = 128 only");
  if (static_cast<int64_t>(B) * H * S_q == 0) return ATTN_OK;  // nothing to compute
  if (!q || !o || (S_kv > 0 && (!k || !v)))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be non-NULL");
  if (!aligned16(q) || !aligned16(o) || (S_kv > 0 && (!aligned16(k) || !aligned16(v))))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  const int64_t elems = static_cast<int64_t>(B) * H * (S_q > S_kv ? S_q : S_kv) * D;
  if (elems * 2 >= (int64_t(1) << 40))
    return fail(ATTN_ERR_UNSUPPORTED, "tensor too large for one TMA descriptor");
  const int rows = attn_sm103a::prefill_rows_per_cta();
  const int64_t n_qb = (S_q + rows - 1) / rows;
  if (static_cast<int64_t>(B) * H * n_qb > 0x7FFFFFFF)
    return fail(ATTN_ERR_UNSUPPORTED, "grid too large");

  DeviceState* st = nullptr;
  attn_status s = device_state(&st);
  if (s != ATTN_OK) return s;

  const bool bshd = layout == ATTN_BSHD;
  CUtensorMap mq, mk, mv, mo;
  const int S_kv_map = S_kv > 0 ? S_kv : 1;
  const void* kb = S_kv > 0 ? k : q;
  const void* vb = S_kv > 0 ? v : q;
  if (!prefill_map_fp8(&mq, q, B, H, S_q, D, bshd) ||
      !prefill_map_fp8(&mk, kb, B, H, S_kv_map, D, bshd) ||
      !prefill_map_fp8(&mv, vb, B, H, S_kv_map, D, bshd) ||
      !prefill_map(&mo, o, B, H, S_q, D, bshd, out_dtype == ATTN_BF16))
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for an FP8 prefill tensor");

  attn_sm103a::PrefillParams p{};
  p.lse = lse;
  p.o_scale = descale_v;
  p.B = B;
  p.H = H;
  p.S_q = S_q;
  p.S_kv = S_kv;
  p.num_q_blocks = static_cast<int>(n_qb);
  p.causal = causal;
  p.bshd = bshd ? 1 : 0;
  // scores of the stored codes times descale_q * descale_k are the real ones
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * descale_q * descale_k *
                                    1.4426950408889634);
  p.err = st->err_word;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.o = o;
  p.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0 ? 1 : 0;
  p.ctas = st->num_sms;
  s = prefill_sched(st, stream, &p.sched);
  if (s != ATTN_OK) return s;
  cudaError_t e =
      attn_sm103a::prefill_fp8_launch(mq, mk, mv, mo, p, out_dtype == ATTN_BF16, stream);
  if (e != cudaSuccess) return fail_cuda(e, "FP8 prefill launch");
  return ATTN_OK;
}

attn_status attn_extend_fwd(const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* page_table, const int32_t* kv_lens, void* o, float* lse,
                            int B, int S_q, int H_q, int H_kv, int D, int page_size,
                            int max_pages_per_seq, int num_pages, attn_dtype dtype, int causal,
                            float scale, cudaStream_t stream) {
  if (B < 0 || S_q < 0) return fail(ATTN_ERR_INVALID_ARG, "B and S_q must be >= 0");
  if (H_q <= 0 || H_kv <= 0) return fail(ATTN_ERR_INVALID_ARG, "H_q and H_kv must be > 0");
  if (H_q % H_kv != 0) return fail(ATTN_ERR_INVALID_ARG, "H_q must be a multiple of H_kv");
  if (D != 64 && D != 128) return fail(ATTN_ERR_UNSUPPORTED, "D must be 64 or 128");
  if (dtype != ATTN_F16 && dtype != ATTN_BF16)
    return fail(ATTN_ERR_INVALID_ARG, "dtype must be ATTN_F16 or ATTN_BF16");
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!(std::isfinite(scale) && scale > 0.f))
    return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (page_size <= 0 || max_pages_per_seq <= 0 || num_pages <= 0)
    return fail(ATTN_ERR_INVALID_ARG, "page_size, max_pages_per_seq and num_pages must be > 0");
  const int tile = attn_sm103a::prefill_box_rows();
  const bool small_ok = page_size >= 8 && page_size <= tile && tile % page_size == 0;
  if (!small_ok && page_size % tile != 0)
    return fail(ATTN_ERR_UNSUPPORTED, "page_size must be 8, 16, 32, 64 or a multiple of 128");
  if (static_cast<int64_t>(B) * S_q == 0) return ATTN_OK;  // nothing to compute
  if (!q || !k_pool || !v_pool || !page_table || !kv_lens || !o)
    return fail(ATTN_ERR_INVALID_ARG,
                "q, k_pool, v_pool, page_table, kv_lens and o must be non-NULL");
  if (!aligned16(q) || !aligned16(o) || !aligned16(k_pool) || !aligned16(v_pool))
    return fail(ATTN_ERR_INVALID_ARG, "q, k_pool, v_pool and o must be 16-byte aligned");
  if (static_cast<int64_t>(max_pages_per_seq) * page_size > 0x7FFFFFFF)
    return fail(ATTN_ERR_UNSUPPORTED, "KV capacity exceeds 2^31 keys");
  if ((static_cast<int64_t>(num_pages) + 1) * page_size > 0x7FFFFFFF)
    return fail(ATTN_ERR_UNSUPPORTED, "KV pool exceeds 2^31 rows");
  if (static_cast<int64_t>(num_pages) * page_size * H_kv * D * 2 >= (int64_t(1) << 40) ||
      static_cast<int64_t>(B) * S_q * H_q * D * 2 >= (int64_t(1) << 40))
    return fail(ATTN_ERR_UNSUPPORTED, "tensor too large for one TMA descriptor");
  const int rows = attn_sm103a::prefill_rows_per_cta();
  const int64_t n_qb = (S_q + rows - 1) / rows;
  if (static_cast<int64_t>(B) * H_q * n_qb > 0x7FFFFFFF)
    return fail(ATTN_ERR_UNSUPPORTED, "grid too large");

  DeviceState* st = nullptr;
  attn_status s = device_state(&st);
  if (s != ATTN_OK) return s;

  const bool bf16 = dtype == ATTN_BF16;
  const int box_rows = page_size < tile ? page_size : tile;
  CUtensorMap mq, mk, mv, mo;
  if (!prefill_map(&mq, q, B, H_q, S_q, D, true, bf16) ||
      !prefill_map(&mo, o, B, H_q, S_q, D, true, bf16) ||
      !extend_map(&mk, k_pool, num_pages, page_size, H_kv, D, box_rows, bf16) ||
      !extend_map(&mv, v_pool, num_pages, page_size, H_kv, D, box_rows, bf16))
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for an extend tensor");

  attn_sm103a::PrefillParams p{};
  p.lse = lse;
  p.o_scale = 1.f;
  p.B = B;
  p.H = H_q;
  p.S_q = S_q;
  p.S_kv = 0;  // per sequence, from kv_lens
  p.num_q_blocks = static_cast<int>(n_qb);
  p.causal = causal;
  p.bshd = 1;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = st->err_word;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.page_table = page_table;
  p.kv_lens = kv_lens;
  p.max_pages = max_pages_per_seq;
  p.page_size = page_size;
  p.num_pages = num_pages;
  p.group = H_q / H_kv;
  p.H_kv = H_kv;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  // Pages of at most 16 keys make the page-box gather the bottleneck: CTA
  // pairs that share a kv head split it (the group must be even).
  p.pair = (p.group % 2 == 0 && page_size <= 16) ? 1 : 0;
  cudaError_t e = attn_sm103a::extend_launch(mq, mk, mv, mo, p, D, bf16, stream);
  if (e != cudaSuccess) return fail_cuda(e, "extend launch");
  return ATTN_OK;
}

attn_status attn_decode_fwd(const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* page_table, const int32_t* kv_lens, void* o, int B,
                            int H_q, int H_kv, int D, int page_size, int max_pages_per_seq,
                            int num_pages, int num_splits, float scale, attn_dtype dtype,
                            cudaStream_t stream) {
  attn_internal::DecodePlan plan;
  attn_status s = attn_internal::decode_plan(q, k_pool, v_pool, page_table, kv_lens, o, B, H_q,
                                             H_kv, D, page_size, max_pages_per_seq, num_pages,
                                             num_splits, scale, dtype, &plan);
  if (s != ATTN_OK || plan.empty) return s;
  DeviceState* st = nullptr;
  s = device_state(&st);
  if (s != ATTN_OK) return s;

  // The stream's workspace.  A graph captured earlier may hold the current
  // buffer's address, so a buffer that has to grow is retired, not freed:
  // retired buffers are freed by attn_release_workspace.  Growth is at least
  // 2x, so retired buffers add up to less than the live one.
  const size_t need = plan.partial_bytes;
  void* workspace = nullptr;
  {
    std::lock_guard<std::mutex> lk(st->mu);
    DeviceState::Workspace& w = st->workspaces[stream];
    if (w.bytes < need) {
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      cudaError_t e = cudaStreamIsCapturing(stream, &cs);
      if (e != cudaSuccess) return fail_cuda(e, "cudaStreamIsCapturing");
      if (cs != cudaStreamCaptureStatusNone)
        return fail(ATTN_ERR_NO_MEMORY,
                    "decode workspace must grow but the stream is capturing; call once before "
                    "capture with the largest shapes");
      const size_t bytes = need > 2 * w.bytes ? need : 2 * w.bytes;
      void* ws = nullptr;
      e = cudaMalloc(&ws, bytes);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(ATTN_ERR_NO_MEMORY, std::string("workspace cudaMalloc: ") + cudaGetErrorString(e));
      }
      if (w.ptr) st->retired.push_back(w.ptr);
      w.ptr = ws;
      w.bytes = bytes;
    }
    workspace = w.ptr;
  }
  return attn_internal::decode_enqueue(plan, static_cast<float*>(workspace), stream);
}

attn_status attn_release_workspace(void) {
  DeviceState* st = nullptr;
  attn_status s = device_state(&st);
  if (s != ATTN_OK) return s;
  std::lock_guard<std::mutex> lk(st->mu);
  if (!st->workspaces.empty() || !st->retired.empty()) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize");
    for (auto& kv : st->workspaces) cudaFree(kv.second.ptr);
    st->workspaces.clear();
    for (void* ptr : st->retired) cudaFree(ptr);
    st->retired.clear();
  }
  if (!st->sched.empty()) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize");
    for (auto& kv : st->sched) cudaFree(kv.second);
    st->sched.clear();
  }
  return ATTN_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------
// The decode plan shared by attn_decode_fwd and attn_decode_fwd_noalloc.
namespace attn_internal {

attn_status set_error(attn_status s, const char* msg) { return fail(s, msg); }

attn_status decode_plan(const void* q, const void* k_pool, const void* v_pool,
                        const int32_t* page_table, const int32_t* kv_lens, void* o, int B,
                        int H_q, int H_kv, int D, int page_size, int max_pages_per_seq,
                        int num_pages, int num_splits, float scale, attn_dtype dtype,
                        DecodePlan* plan) {
  if (B < 0) return fail(ATTN_ERR_INVALID_ARG, "B must be >= 0");
  if (H_q <= 0 || H_kv <= 0) return fail(ATTN_ERR_INVALID_ARG, "H_q and H_kv must be > 0");
  if (H_q % H_kv != 0) return fail(ATTN_ERR_INVALID_ARG, "H_q must be a multiple of H_kv");
  if (H_q / H_kv > 16) return fail(ATTN_ERR_UNSUPPORTED, "H_q / H_kv must be <= 16");
  if (D != 64 && D != 128) return fail(ATTN_ERR_UNSUPPORTED, "D must be 64 or 128");
  if (dtype != ATTN_F16 && dtype != ATTN_BF16)
    return fail(ATTN_ERR_INVALID_ARG, "dtype must be ATTN_F16 or ATTN_BF16");
  if (!(std::isfinite(scale) && scale > 0.f))
    return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (num_splits < 0) return fail(ATTN_ERR_INVALID_ARG, "num_splits must be >= 0");
  if (page_size <= 0) return fail(ATTN_ERR_INVALID_ARG, "page_size must be > 0");
  const bool paged = page_table != nullptr;
  if (paged) {
    if (max_pages_per_seq <= 0 || num_pages <= 0)
      return fail(ATTN_ERR_INVALID_ARG, "max_pages_per_seq and num_pages must be > 0");
    const bool small_ok = page_size <= 64 && 64 % page_size == 0 && page_size >= 8;
    if (!small_ok && page_size % 64 != 0)
      return fail(ATTN_ERR_UNSUPPORTED, "page_size must be 8, 16, 32 or a multiple of 64");
  } else {
    max_pages_per_seq = 1;
    if (num_pages != B)
      return fail(ATTN_ERR_INVALID_ARG, "contiguous cache: num_pages must equal B");
  }
  plan->empty = B == 0;
  if (B == 0) return ATTN_OK;
  if (!q || !k_pool || !v_pool || !kv_lens || !o)
    return fail(ATTN_ERR_INVALID_ARG, "q, k_pool, v_pool, kv_lens and o must be non-NULL");
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(o))
    return fail(ATTN_ERR_INVALID_ARG, "q, k_pool, v_pool and o must be 16-byte aligned");
  const int64_t cap = static_cast<int64_t>(max_pages_per_seq) * page_size;
  if (cap > 0x7FFFFFFF) return fail(ATTN_ERR_UNSUPPORTED, "KV capacity exceeds 2^31 keys");
  if (static_cast<int64_t>(num_pages) * page_size * H_kv * D * 2 >= (int64_t(1) << 40))
    return fail(ATTN_ERR_UNSUPPORTED, "KV pool too large for one TMA descriptor");

  DeviceState* st = nullptr;
  attn_status s = device_state(&st);
  if (s != ATTN_OK) return s;

  // Split plan.  num_splits > 0 splits every sequence into that many parts;
  // 0 fixes a chunk length so that the expected work (sequences assumed half
  // full on average) spans several waves of resident CTAs.
  const int kt = attn_sm103a::decode_keys_per_tile();
  int fixed_chunk = 0, max_splits = 0;
  if (num_splits > 0) {
    max_splits = num_splits;
  } else {
    int chunk = env_int("ATTN_DECODE_SPLIT_CHUNK", 0);
    if (chunk <= 0) {
      const double est_keys = static_cast<double>(B) * H_kv * (static_cast<double>(cap) / 2.0);
      const double target_ctas = 8.0 * 2.0 * st->num_sms;
      chunk = static_cast<int>(est_keys / target_ctas);
      if (chunk < 256) chunk = 256;
      if (chunk > 8192) chunk = 8192;
    }
    chunk = (chunk + kt - 1) / kt * kt;
    fixed_chunk = chunk;
    max_splits = static_cast<int>((cap + chunk - 1) / chunk);
    if (max_splits < 1) max_splits = 1;
  }
  if (static_cast<int64_t>(max_splits) > 65535)
    return fail(ATTN_ERR_UNSUPPORTED, "too many splits for one launch");

  const bool bf16 = dtype == ATTN_BF16;
  const int box_rows = paged ? (page_size < kt ? page_size : kt) : kt;
  const int pages = paged ? num_pages : B;
  if (!decode_map(&plan->mk, k_pool, pages, page_size, H_kv, D, box_rows, bf16) ||
      !decode_map(&plan->mv, v_pool, pages, page_size, H_kv, D, box_rows, bf16))
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the KV pool");

  // Partials: o_part [B, H_q, max_splits, D] then lse_part [B, H_q, max_splits].
  const size_t rows = static_cast<size_t>(B) * H_q * max_splits;
  plan->partial_bytes = rows * (D + 1) * sizeof(float);
  plan->D = D;
  plan->bf16 = bf16;
  plan->o = o;
  attn_sm103a::DecodeParams& p = plan->p;
  p.q = q;
  p.page_table = page_table;
  p.kv_lens = kv_lens;
  p.B = B;
  p.H_q = H_q;
  p.group = H_q / H_kv;
  p.page_size = page_size;
  p.max_pages = max_pages_per_seq;
  p.num_pages = pages;
  p.max_splits = max_splits;
  p.fixed_chunk = fixed_chunk;
  p.num_splits = num_splits > 0 ? num_splits : 1;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = st->err_word;
  p.wait_limit_ns = g_wait_limit_ns.load();
  return ATTN_OK;
}

attn_status decode_enqueue(DecodePlan& plan, float* partials, cudaStream_t stream) {
  const size_t rows = static_cast<size_t>(plan.p.B) * plan.p.H_q * plan.p.max_splits;
  plan.p.o_part = partials;
  plan.p.lse_part = partials + rows * plan.D;
  cudaError_t e = attn_sm103a::decode_launch(plan.mk, plan.mv, plan.p, plan.o, plan.D,
                                             plan.bf16, stream);
  if (e != cudaSuccess) return fail_cuda(e, "decode launch");
  return ATTN_OK;
}

}  // namespace attn_internal
