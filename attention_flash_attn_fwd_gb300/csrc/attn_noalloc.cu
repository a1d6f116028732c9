// attn_noalloc.cu -- attn_decode_fwd_noalloc: decode attention that never
// allocates device memory.
//
// attn_decode_fwd keeps its split partials in a workspace that it grows with
// cudaMalloc.  Some callers cannot let a library allocate: code that is being
// recorded into a CUDA graph (cudaMalloc is not a capturable operation, and a
// mid-capture allocation invalidates the capture), engines whose framework
// owns every byte of device memory through its own pool and budget, and
// latency-critical serving loops that must not block on the allocator or risk
// an out-of-memory error at step time.  For them this entry point puts the
// split partials in one fixed, file-scope device array instead.
//
// The array is kNoAllocScratchBytes (16 MiB) and lives in the library's module
// on every GPU that loads the library, until the process exits.  A call whose
// split plan needs more than that is rejected with ATTN_ERR_UNSUPPORTED.
//
// Every call shares the array and it keeps the last call's contents.  Nothing
// in it has to start at zero: each split writes all of its own partial slots
// (an empty split writes -inf) before the combine kernel, queued after it on
// the same stream, reads them.  Two calls whose kernels overlap on the GPU
// (different streams, or different host threads) race on the array.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <string>

#include "../../include/attn_gb300.h"
#include "decode_sm103a.h"

namespace attn_internal {
attn_status device_info(int** err_word, int* num_sms);
attn_status set_error(attn_status s, const char* msg);
bool encode_decode_map(CUtensorMap* m, const void* base, int num_pages, int page_size, int H_kv,
                       int D, int box_rows, bool bf16);
uint64_t wait_limit_ns();
int split_chunk_override();
}  // namespace attn_internal

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

attn_status bad(attn_status s, const char* msg) { return attn_internal::set_error(s, msg); }

}  // namespace

extern "C" ATTN_API attn_status attn_decode_fwd_noalloc(
    const void* q, const void* k_pool, const void* v_pool, const int32_t* page_table,
    const int32_t* kv_lens, void* o, int B, int H_q, int H_kv, int D, int page_size,
    int max_pages_per_seq, int num_pages, int num_splits, float scale, attn_dtype dtype,
    cudaStream_t stream) {
  // Same argument rules as attn_decode_fwd.
  if (B < 0) return bad(ATTN_ERR_INVALID_ARG, "B must be >= 0");
  if (H_q <= 0 || H_kv <= 0) return bad(ATTN_ERR_INVALID_ARG, "H_q and H_kv must be > 0");
  if (H_q % H_kv != 0) return bad(ATTN_ERR_INVALID_ARG, "H_q must be a multiple of H_kv");
  if (H_q / H_kv > 16) return bad(ATTN_ERR_UNSUPPORTED, "H_q / H_kv must be <= 16");
  if (D != 64 && D != 128) return bad(ATTN_ERR_UNSUPPORTED, "D must be 64 or 128");
  if (dtype != ATTN_F16 && dtype != ATTN_BF16)
    return bad(ATTN_ERR_INVALID_ARG, "dtype must be ATTN_F16 or ATTN_BF16");
  if (!(std::isfinite(scale) && scale > 0.f))
    return bad(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (num_splits < 0) return bad(ATTN_ERR_INVALID_ARG, "num_splits must be >= 0");
  if (page_size <= 0) return bad(ATTN_ERR_INVALID_ARG, "page_size must be > 0");
  const bool paged = page_table != nullptr;
  if (paged) {
    if (max_pages_per_seq <= 0 || num_pages <= 0)
      return bad(ATTN_ERR_INVALID_ARG, "max_pages_per_seq and num_pages must be > 0");
    const bool small_ok = page_size <= 64 && 64 % page_size == 0 && page_size >= 8;
    if (!small_ok && page_size % 64 != 0)
      return bad(ATTN_ERR_UNSUPPORTED, "page_size must be 8, 16, 32 or a multiple of 64");
  } else {
    max_pages_per_seq = 1;
    if (num_pages != B) return bad(ATTN_ERR_INVALID_ARG, "contiguous cache: num_pages must equal B");
  }
  if (B == 0) return ATTN_OK;
  if (!q || !k_pool || !v_pool || !kv_lens || !o)
    return bad(ATTN_ERR_INVALID_ARG, "q, k_pool, v_pool, kv_lens and o must be non-NULL");
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!a16(q) || !a16(k_pool) || !a16(v_pool) || !a16(o))
    return bad(ATTN_ERR_INVALID_ARG, "q, k_pool, v_pool and o must be 16-byte aligned");
  const int64_t cap = static_cast<int64_t>(max_pages_per_seq) * page_size;
  if (cap > 0x7FFFFFFF) return bad(ATTN_ERR_UNSUPPORTED, "KV capacity exceeds 2^31 keys");
  if (static_cast<int64_t>(num_pages) * page_size * H_kv * D * 2 >= (int64_t(1) << 40))
    return bad(ATTN_ERR_UNSUPPORTED, "KV pool too large for one TMA descriptor");

  int* err_word = nullptr;
  int num_sms = 0;
  attn_status s = attn_internal::device_info(&err_word, &num_sms);
  if (s != ATTN_OK) return s;

  // Same split plan as attn_decode_fwd.
  const int kt = attn_sm103a::decode_keys_per_tile();
  int fixed_chunk = 0, max_splits = 0;
  if (num_splits > 0) {
    max_splits = num_splits;
  } else {
    int chunk = attn_internal::split_chunk_override();
    if (chunk <= 0) {
      const double est_keys = static_cast<double>(B) * H_kv * (static_cast<double>(cap) / 2.0);
      chunk = static_cast<int>(est_keys / (8.0 * 2.0 * num_sms));
      if (chunk < 256) chunk = 256;
      if (chunk > 8192) chunk = 8192;
    }
    chunk = (chunk + kt - 1) / kt * kt;
    fixed_chunk = chunk;
    max_splits = static_cast<int>((cap + chunk - 1) / chunk);
    if (max_splits < 1) max_splits = 1;
  }
  if (max_splits > 65535) return bad(ATTN_ERR_UNSUPPORTED, "too many splits for one launch");

  const size_t rows = static_cast<size_t>(B) * H_q * max_splits;
  const size_t need = rows * (D + 1) * sizeof(float);
  if (need > kNoAllocScratchBytes) {
    std::string msg = "attn_decode_fwd_noalloc needs " + std::to_string(need) +
                      " bytes of split scratch but its fixed array holds " +
                      std::to_string(kNoAllocScratchBytes) +
                      "; use fewer splits (num_splits), a smaller batch, or attn_decode_fwd";
    return bad(ATTN_ERR_UNSUPPORTED, msg.c_str());
  }
  float* scratch = nullptr;
  s = scratch_for_current_device(&scratch);
  if (s != ATTN_OK) return s;

  const bool bf16 = dtype == ATTN_BF16;
  const int box_rows = paged ? (page_size < kt ? page_size : kt) : kt;
  CUtensorMap mk, mv;
  const int pages = paged ? num_pages : B;
  if (!attn_internal::encode_decode_map(&mk, k_pool, pages, page_size, H_kv, D, box_rows, bf16) ||
      !attn_internal::encode_decode_map(&mv, v_pool, pages, page_size, H_kv, D, box_rows, bf16))
    return bad(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the KV pool");

  attn_sm103a::DecodeParams p{};
  p.q = q;
  p.page_table = page_table;
  p.kv_lens = kv_lens;
  p.o_part = scratch;
  p.lse_part = scratch + rows * D;
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
  p.err = err_word;
  p.wait_limit_ns = attn_internal::wait_limit_ns();
  cudaError_t e = attn_sm103a::decode_launch(mk, mv, p, o, D, bf16, stream);
  if (e != cudaSuccess) {
    std::string msg = std::string("decode launch: ") + cudaGetErrorString(e);
    return bad(ATTN_ERR_CUDA, msg.c_str());
  }
  return ATTN_OK;
}
