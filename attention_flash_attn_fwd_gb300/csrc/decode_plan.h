// decode_plan.h -- the decode entry points' shared argument checks, split plan
// and launch (library-internal; not part of the C ABI).
//
// attn_decode_fwd (partials in a per-stream workspace it allocates) and
// attn_decode_fwd_noalloc (partials in a fixed device array) differ only in
// where the split partials live.  Both call decode_plan() and
// decode_enqueue(), so they validate the same way, pick the same split plan
// and launch the same kernels: for equal inputs their outputs are bitwise
// equal.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/attn_gb300.h"
#include "decode_sm103a.h"

namespace attn_internal {

struct DecodePlan {
  bool empty = false;           // B == 0: nothing to launch
  int D = 0;
  bool bf16 = false;
  void* o = nullptr;
  size_t partial_bytes = 0;     // split partials: B * H_q * max_splits * (D + 1) fp32
  CUtensorMap mk{}, mv{};       // K and V pool tensor maps
  attn_sm103a::DecodeParams p{};  // all but o_part / lse_part
};

// Validates attn_decode_fwd's arguments (same rules, same error codes and
// messages) and computes the split plan; launches nothing.
attn_status decode_plan(const void* q, const void* k_pool, const void* v_pool,
                        const int32_t* page_table, const int32_t* kv_lens, void* o, int B,
                        int H_q, int H_kv, int D, int page_size, int max_pages_per_seq,
                        int num_pages, int num_splits, float scale, attn_dtype dtype,
                        DecodePlan* plan);

// Enqueues the split and combine kernels of `plan` on `stream` with the split
// partials at `partials` (plan.partial_bytes bytes, 16-byte aligned).
attn_status decode_enqueue(DecodePlan& plan, float* partials, cudaStream_t stream);

// Records `msg` as the calling thread's last error and returns `s`.
attn_status set_error(attn_status s, const char* msg);

}  // namespace attn_internal
