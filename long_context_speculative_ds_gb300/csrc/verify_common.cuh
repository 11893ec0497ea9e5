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

// Output row r of a row group merged over the group's ns splits (items
// base .. base + ns - 1): sum over s of 2^{lse_s - lse} O_s, the split
// outputs O_s being normalised and lse the row's final log2-sum-exp.  One
// warp, lane-parallel over columns; the split log2-sum-exps are loaded
// lane-parallel over splits and the weights broadcast from the lane that
// holds split s.  NB splits per round trip.  Split outputs are bf16 (HALF)
// or f32; the result goes to out row out_row ([n_nodes * num_q_heads] rows
// of head_dim) in the output dtype.
template <int D, bool HALF, int NB>
DS_DEV void combine_row_splits(const VerifyKArgs& a, int64_t base, int ns, int r, float lse,
                               int64_t out_row) {
  static_assert(NB <= 32, "split weights are held one per lane");
  const int lane = threadIdx.x & 31;
  const float* lp = a.lse_part + base * kRowsPerGroup + r;
  constexpr int E = D / 32;                  // columns per lane (4 or 2)
  constexpr int W = HALF ? E / 2 : E;        // 32-bit words per lane and split
  constexpr int kWordsPerRow = HALF ? D / 2 : D;
  const uint32_t* op0 = reinterpret_cast<const uint32_t*>(a.o_part) +
                        (base * kRowsPerGroup + r) * kWordsPerRow + lane * W;
  constexpr int64_t sstride = (int64_t)kRowsPerGroup * kWordsPerRow;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int s0 = 0; s0 < ns; s0 += NB) {
    uint32_t x[NB][W];
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      if (s0 + k < ns) {
        const uint32_t* op = op0 + (s0 + k) * sstride;
        if constexpr (W == 4) {
          const uint4 v = __ldcg(reinterpret_cast<const uint4*>(op));
          x[k][0] = v.x; x[k][1] = v.y; x[k][2] = v.z; x[k][3] = v.w;
        } else if constexpr (W == 2) {
          const uint2 v = __ldcg(reinterpret_cast<const uint2*>(op));
          x[k][0] = v.x; x[k][1] = v.y;
        } else {
          x[k][0] = __ldcg(op);
        }
      }
    }
    const float wl = (lane < NB && s0 + lane < ns)
                         ? exp2f(__ldcg(lp + (int64_t)(s0 + lane) * kRowsPerGroup) - lse)
                         : 0.f;
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const float w = __shfl_sync(0xffffffffu, wl, k);
      if (s0 + k < ns && w != 0.f) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          float xv;
          if constexpr (HALF)   // bf16 pair: element 2i in the low half
            xv = __uint_as_float((e & 1) ? (x[k][e >> 1] & 0xffff0000u) : (x[k][e >> 1] << 16));
          else
            xv = __uint_as_float(x[k][e]);
          acc[e] = fmaf(w, xv, acc[e]);
        }
      }
    }
  }
  const int64_t obase = out_row * D + lane * E;
  if (a.out_f32) {
    float* out = reinterpret_cast<float*>(a.out) + obase;
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = acc[e];
  } else {
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) + obase;
#pragma unroll
    for (int e = 0; e < E; e += 2)
      *reinterpret_cast<__nv_bfloat162*>(out + e) = __floats2bfloat162_rn(acc[e], acc[e + 1]);
  }
}

}  // namespace ds
