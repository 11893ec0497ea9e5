// Kernel arguments shared by the split-pass, combine and finalize kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "dev_common.cuh"

namespace ds {

struct VerifyKArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* page_table;
  const int32_t* parents;
  PlanArgs plan;
  int32_t num_q_heads, num_pages;
  int64_t page_stride, tok_stride, head_stride;   // elements
  float scale_log2;
  uint32_t* counters;
  int4* gdesc;
  float* o_part;
  float* lse_part;
  float* clse;
  float* row_lse;
  void* out;
  int32_t out_f32;
  float* scores;
  int32_t accumulate;
};

}  // namespace ds
