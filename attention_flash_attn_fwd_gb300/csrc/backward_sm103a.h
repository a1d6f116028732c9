// backward_sm103a.h -- launch interface of the attention backward kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn_sm103a {

struct BackwardParams {
  const void* o;          // forward output, q's layout, 16-bit
  const void* dout;       // upstream gradient, q's layout, 16-bit
  const float* lse;       // [B, H, S_q] natural-log row sums of the forward
  float* delta;           // [B, H, S_q] scratch: rowsum(dO * O)
  int B, H, S_q, S_kv;
  int causal;             // bottom-right aligned causal mask
  int bshd;               // 1: [B,S,H,D]; 0: [B,H,S,D]
  float scale;            // softmax scale
  float scale_log2;       // scale * log2(e)
  int* err;               // device error word
  uint64_t wait_limit_ns; // bound on every mbarrier wait
};

// D = 128 only.  Maps: 16-bit, 128-byte swizzle, box 64 columns x 128 rows,
// the prefill layout (BHSD (D, S, H, B), BSHD (D, H, S, B)).
cudaError_t backward_launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dout, const CUtensorMap& dq, const CUtensorMap& dk,
                            const CUtensorMap& dv, const BackwardParams& p, bool bf16,
                            cudaStream_t stream);

}  // namespace attn_sm103a
