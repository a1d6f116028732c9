// mqa_logits_sm103a.h -- launch interface of the FP8 MQA logits kernel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn_sm103a {

struct MqaParams {
  const float* kv_scale;   // [S_kv]
  const float* w;          // [S_q, H]
  const int32_t* start;    // [S_q] window starts
  const int32_t* end;      // [S_q] window ends (exclusive)
  float* logits;           // [S_q, stride]
  int64_t stride;          // row stride of logits, >= S_kv
  int S_q, S_kv, H;        // H in {32, 64, 128}; D = 128
  int clean;               // 1: -inf outside the window
  int groups_per_cta;      // query groups each CTA walks
  int* err;                // device error word
  uint64_t wait_limit_ns;  // bound on every mbarrier wait
};

// q map: E4M3 [S_q * H, 128] as 2-D, box 128 x 256 rows, 128-byte swizzle;
// k map: E4M3 [S_kv, 128] as 2-D, box 128 x 128 rows, 128-byte swizzle.
cudaError_t mqa_logits_launch(const CUtensorMap& q, const CUtensorMap& k, const MqaParams& p,
                              cudaStream_t stream);
int mqa_rows_per_group(int H);
int mqa_keys_per_cta();

}  // namespace attn_sm103a
