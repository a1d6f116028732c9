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
  int tiles_per_cta;       // 128-key tiles each CTA walks
  int* err;                // device error word
  uint64_t wait_limit_ns;  // bound on every mbarrier wait
};

// q map: E4M3 [S_q * H, 128] as 2-D, box 128 x mqa_rows_per_slab_box() rows;
// k map: E4M3 [S_kv, 128] as 2-D, box 128 x mqa_keys_per_tile() rows; both
// with 128-byte swizzle.  The grid is (query blocks of mqa_rows_per_block(H)
// rows) x (key splits of p.tiles_per_cta tiles).
cudaError_t mqa_logits_launch(const CUtensorMap& q, const CUtensorMap& k, const MqaParams& p,
                              cudaStream_t stream);
int mqa_rows_per_block(int H);
int mqa_keys_per_tile();
int mqa_rows_per_slab_box();
// Tiles per CTA that balance the grid over num_sms SMs.
int mqa_tiles_per_cta(int S_q, int S_kv, int H, int num_sms);

}  // namespace attn_sm103a
