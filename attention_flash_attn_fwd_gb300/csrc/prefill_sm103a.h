// prefill_sm103a.h -- launch interface of the prefill attention kernel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn_sm103a {

struct PrefillParams {
  float* lse;             // [B, H, S_q] natural-log row sums, or nullptr
  int B, H, S_q, S_kv;
  int num_q_blocks;       // ceil(S_q / prefill_rows_per_cta())
  int causal;             // bottom-right aligned causal mask
  int bshd;               // 1: tensor maps are (D, H, S, B); 0: (D, S, H, B)
  float scale_log2;       // softmax scale * log2(e)
  int* err;               // device error word
  uint64_t wait_limit_ns; // bound on every mbarrier wait
  // Paged K/V (extend form only; unused by the contiguous prefill):
  const int32_t* page_table;  // [B, max_pages] physical page ids
  const int32_t* kv_lens;     // [B] keys per sequence (S_kv is ignored)
  int max_pages, page_size, num_pages;
  int group;                  // query heads per kv head (H / H_kv)
  int H_kv;
  const void* k_pool;         // [num_pages, page_size, H_kv, D]
  const void* v_pool;
  int pair;                   // 1: CTA pairs (clusters of 2) share K/V tiles; needs an even group
  float o_scale;              // multiplies O at the end (the FP8 form's V descale, else 1)
  // Contiguous forms only:
  void* o;                    // O, 16-bit, q's layout (stored directly by the softmax warps)
  int* sched;                 // zeroed unit counter: persistent CTAs; nullptr: one CTA per unit
  int ctas;                   // persistent CTAs to launch (the SM count)
  int o_align32;              // o is 32-byte aligned: whole-sector stores
};

// Tensor maps: 16-bit elements, 128-byte swizzle, box = 64 columns x
// prefill_box_rows() rows of one (batch, head).
cudaError_t prefill_launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const CUtensorMap& o, const PrefillParams& p, int D, bool bf16,
                           cudaStream_t stream);

// Extend form: q/o maps as BSHD (D, H, S_q, B); k/v maps over the pool
// [num_pages, page_size, H_kv, D] as 2-D (H_kv * D, num_pages * page_size)
// with box (64, min(page_size, 128)).
cudaError_t extend_launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& o, const PrefillParams& p, int D, bool bf16,
                          cudaStream_t stream);

// FP8 form (D = 128 only): q/k/v maps over E4M3 bytes, box 128 columns x
// prefill_box_rows() rows; o map 16-bit as for prefill.
cudaError_t prefill_fp8_launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& o, const PrefillParams& p, bool bf16_out,
                               cudaStream_t stream);

int prefill_rows_per_cta();
int prefill_box_rows();

}  // namespace attn_sm103a
