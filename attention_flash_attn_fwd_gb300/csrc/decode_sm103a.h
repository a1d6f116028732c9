// decode_sm103a.h -- launch interface of the split-KV decode kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn_sm103a {

struct DecodeParams {
  const void* q;              // [B, H_q, D] 16-bit
  const int32_t* page_table;  // [B, max_pages] or nullptr (contiguous cache)
  const int32_t* kv_lens;     // [B]
  float* o_part;              // [B, H_q, max_splits, D] normalised split outputs
  float* lse_part;            // [B, H_q, max_splits] log2-sum-exp of each split
  int B, H_q, group;          // group = H_q / H_kv query heads per kv head
  int page_size, max_pages, num_pages;
  int max_splits;             // grid extent along splits
  int fixed_chunk;            // > 0: keys per split; 0: derived from num_splits
  int num_splits;             // used when fixed_chunk == 0
  float scale_log2;           // softmax scale * log2(e)
  int* err;                   // device error word
  uint64_t wait_limit_ns;     // bound on every mbarrier wait
};

// Tensor maps over the K and V pools: dims (D, H_kv, page_size, num_pages),
// 16-bit, 128-byte swizzle, box (64, 1, min(page_size, 64) or 64, 1).
cudaError_t decode_launch(const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p,
                          void* out, int D, bool bf16, cudaStream_t stream);

int decode_keys_per_tile();

}  // namespace attn_sm103a
