// attn_noalloc.cu -- attn_decode_fwd_noalloc: decode attention that never
// allocates device memory.
//
// attn_decode_fwd keeps its split partials in a workspace that it grows with
// cudaMalloc.  Some callers cannot let a library allocate: engines whose
// framework owns every byte of device memory through its own pool and budget
// (a library cudaMalloc there either fails, because the pool has already
// reserved the memory, or escapes the framework's accounting), and serving
// loops that must not block on the allocator or risk an out-of-memory error
// in the middle of a step.  For them this entry point puts the split partials
// in one fixed, file-scope device array instead; everything else (checks,
// split plan, kernels) is attn_decode_fwd's own, through one shared helper.
//
// The array is kNoAllocScratchBytes (16 MiB) and lives in the library's module
// on every GPU that loads the library, until the process exits.  A call whose
// split plan needs more than that is rejected with ATTN_ERR_UNSUPPORTED before
// anything is launched.  The first call on a device looks up the array's
// device address with cudaGetSymbolAddress (host code cannot use the array's
// name as a device pointer); make that first call before any stream capture.
//
// Every call shares the array and it keeps the last call's contents.  Nothing
// in it has to start at zero: each split writes all of its own partial slots
// (an empty split writes -inf) before the combine kernel, queued after it on
// the same stream, reads them.  Two calls whose kernels overlap on the GPU
// (different streams, or different host threads) race on the array.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <string>

#include "../../include/attn_gb300.h"
#include "decode_plan.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).
attn_status scratch_for_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return attn_internal::set_error(ATTN_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices)
    return attn_internal::set_error(ATTN_ERR_UNSUPPORTED, "device index too large");
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    float* ptr = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      std::string msg = std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e);
      return attn_internal::set_error(ATTN_ERR_CUDA, msg.c_str());
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" ATTN_API attn_status attn_decode_fwd_noalloc(
    const void* q, const void* k_pool, const void* v_pool, const int32_t* page_table,
    const int32_t* kv_lens, void* o, int B, int H_q, int H_kv, int D, int page_size,
    int max_pages_per_seq, int num_pages, int num_splits, float scale, attn_dtype dtype,
    cudaStream_t stream) {
  // The same checks and split plan as attn_decode_fwd (one shared helper).
  attn_internal::DecodePlan plan;
  attn_status s = attn_internal::decode_plan(q, k_pool, v_pool, page_table, kv_lens, o, B, H_q,
                                             H_kv, D, page_size, max_pages_per_seq, num_pages,
                                             num_splits, scale, dtype, &plan);
  if (s != ATTN_OK || plan.empty) return s;
  if (plan.partial_bytes > kNoAllocScratchBytes) {
    std::string msg = "attn_decode_fwd_noalloc needs " + std::to_string(plan.partial_bytes) +
                      " bytes of split scratch but its fixed array holds " +
                      std::to_string(kNoAllocScratchBytes) +
                      "; use fewer splits (num_splits), a smaller batch, or attn_decode_fwd";
    return attn_internal::set_error(ATTN_ERR_UNSUPPORTED, msg.c_str());
  }
  float* scratch = nullptr;
  s = scratch_for_current_device(&scratch);
  if (s != ATTN_OK) return s;
  return attn_internal::decode_enqueue(plan, scratch, stream);
}
