// Tree-verify attention over a paged bf16 KV cache with fused chunk salience.
//
// Two launches per call:
//   1. split pass   (tcgen05 kernel in verify_tc.cu) one CTA per work item
//                   (sequence, kv head, row group, split of key tiles):
//                   online softmax over its key tiles, writing
//                   the split's normalised output, its row log2-sum-exp, and
//                   for every context chunk in its range the chunk's log2
//                   attention mass per row (log2 sum_{t in chunk} 2^{s_t});
//                   the last split of each row group to finish also forms
//                   the rows' final log2-sum-exp.
//   2. finish       in one grid, independently:
//                   combine: log-sum-exp merge of the splits of each row ->
//                   out;
//                   finalize: chunk score = sum over rows of 2^{chunk mass -
//                   row lse}, the mass under the full softmax denominator,
//                   summed over all query heads and nodes (vllm-diffspec
//                   README, "Architecture": chunks scored from paged target
//                   KV).
// Scores are carried in log2 units (s * scale * log2 e) throughout.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "dev_common.cuh"
#include "internal.h"
#include "pdl.cuh"
#include "verify_common.cuh"

namespace ds {

// ---------------------------------------------------------------------------
// finish: one launch, two independent jobs, both reading the split pass's
// outputs and the final row log2-sum-exp that the last split of each row
// group formed.
//
// combine (the first n_comb CTAs): one warp per (sequence, kv head, row
//   group, row).  The sequence's sizes and the row group's descriptor (its
//   first split item and split count, written by its last split) come in one
//   round trip; then the outputs of kCombBatch splits at a time (lane-
//   parallel over columns) together with their log2-sum-exps (lane-parallel
//   over splits) and the row's final log2-sum-exp; the weights 2^{lse_s -
//   lse} are broadcast from the lane that holds split s.  The batch keeps the
//   kernel within 64 registers, so that every CTA of the launch is resident
//   at once.
// finalize (the rest): one warp per (chunk, sequence).  Lane i covers rows
//   4i .. 4i + 3 and 128 + 4i .. 128 + 4i + 3 of every (kv head, row group)
//   with 16-byte loads; kFinCombos (kv head, row group) combinations per
//   round.
constexpr int kCombBatch = 8;
constexpr int kFinCombos = 3;   // (kv head, row group) combinations per finalize round
constexpr int kFinishThreads = 256;
constexpr int kFinishWarps = kFinishThreads / 32;

template <int D>
DS_DEV void combine_row(const VerifyKArgs& a, int blk) {
  const int row_blocks = kRowsPerGroup / kFinishWarps;
  const int grp = blk / row_blocks, rblk = blk % row_blocks;
  const int per_b = a.plan.num_kv_heads * a.plan.rg_max;
  const int b = grp / per_b;
  const int h = (grp / a.plan.rg_max) % a.plan.num_kv_heads;
  const int rgi = grp % a.plan.rg_max;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = rblk * kFinishWarps + warp;
  // sizes, descriptor and the row's final log2-sum-exp in one round trip
  const SeqPlan sq = seq_sizes(a.plan, b, false);
  const int4 gd = __ldcg(a.gdesc + grp);
  const float lse = __ldcg(a.row_lse + (int64_t)grp * kRowsPerGroup + r);
  if (sq.T == 0 || rgi >= sq.rg) return;
  const int rows_here = min(kRowsPerGroup, sq.rows - rgi * kRowsPerGroup);
  if (r >= rows_here) return;
  const int G = a.plan.group;
  const int grow = rgi * kRowsPerGroup + r;
  const int node = sq.node0 + grow / G;
  const int qh = h * G + grow % G;
  const int base = gd.x;
  const int ns = gd.y;
  const float* lp = a.lse_part + (int64_t)base * kRowsPerGroup + r;
  constexpr int E = D / 32;   // floats per lane (4 or 2)
  const float* op0 = a.o_part + ((int64_t)base * kRowsPerGroup + r) * D + lane * E;
  const int64_t sstride = (int64_t)kRowsPerGroup * D;

  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int s0 = 0; s0 < ns; s0 += kCombBatch) {
    float x[kCombBatch][E];
#pragma unroll
    for (int k = 0; k < kCombBatch; ++k) {
      if (s0 + k < ns) {
        const float* op = op0 + (int64_t)(s0 + k) * sstride;
        if constexpr (E == 4) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(op));
          x[k][0] = v.x; x[k][1] = v.y; x[k][2] = v.z; x[k][3] = v.w;
        } else {
          const float2 v = __ldcg(reinterpret_cast<const float2*>(op));
          x[k][0] = v.x; x[k][1] = v.y;
        }
      }
    }
    // weight of split s0 + lane (lanes below kCombBatch), broadcast below
    const float wl = (lane < kCombBatch && s0 + lane < ns)
                         ? exp2f(__ldcg(lp + (int64_t)(s0 + lane) * kRowsPerGroup) - lse)
                         : 0.f;
#pragma unroll
    for (int k = 0; k < kCombBatch; ++k) {
      const float w = __shfl_sync(0xffffffffu, wl, k);
      if (s0 + k < ns && w != 0.f) {
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(w, x[k][e], acc[e]);
      }
    }
  }
  const int64_t obase = ((int64_t)node * a.num_q_heads + qh) * D + lane * E;
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

DS_DEV void finalize_chunk(const VerifyKArgs& a, int blk) {
  const int nblk_b = (a.plan.max_chunks + kFinishWarps - 1) / kFinishWarps;
  const int b = blk / nblk_b;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = (blk % nblk_b) * kFinishWarps + warp;
  if (c >= a.plan.max_chunks) return;
  static_assert(kRowsPerGroup == 256, "two 128-row halves of four rows per lane");
  // Combinations are enumerated over the workspace's fixed (kv head, row
  // group) layout, so the first round's loads are issued together with the
  // sequence's sizes; combinations and rows the sequence does not have are
  // masked once the sizes are known.
  const int rg_max = a.plan.rg_max;
  const int combos = a.plan.num_kv_heads * rg_max;
  float4 v[kFinCombos][2], w[kFinCombos][2];
  auto load = [&](int cb0) {
#pragma unroll
    for (int k = 0; k < kFinCombos; ++k) {
      if (cb0 + k < combos) {
        const int64_t hb = (int64_t)b * combos + cb0 + k;
        const float4* cl = reinterpret_cast<const float4*>(
            a.clse + (hb * a.plan.max_chunks + c) * kRowsPerGroup);
        const float4* rl = reinterpret_cast<const float4*>(a.row_lse + hb * kRowsPerGroup);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          v[k][q] = __ldcg(cl + lane + 32 * q);
          w[k][q] = __ldg(rl + lane + 32 * q);
        }
      }
    }
  };
  load(0);
  const SeqPlan sq = seq_sizes(a.plan, b, false);
  const int n_ch = (sq.L + a.plan.chunk_size - 1) / a.plan.chunk_size;
  if (c >= n_ch) return;
  float sum = 0.f;
  for (int cb0 = 0; cb0 < combos; cb0 += kFinCombos) {
    if (cb0 > 0) load(cb0);
#pragma unroll
    for (int k = 0; k < kFinCombos; ++k) {
      const int rgi = (cb0 + k) % rg_max;
      if (cb0 + k < combos && rgi < sq.rg) {
        const int rows_here = min(kRowsPerGroup, sq.rows - rgi * kRowsPerGroup);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int r0 = 4 * lane + 128 * q;
          const float vv[4] = {v[k][q].x, v[k][q].y, v[k][q].z, v[k][q].w};
          const float ww[4] = {w[k][q].x, w[k][q].y, w[k][q].z, w[k][q].w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (r0 + e < rows_here) sum += exp2f(vv[e] - ww[e]);
        }
      }
    }
  }
  sum = warp_sum(sum);
  if (lane == 0) {
    float* dst = a.scores + (int64_t)b * a.plan.max_chunks + c;
    *dst = a.accumulate ? *dst + sum : sum;
  }
}

template <int D>
__global__ void __launch_bounds__(kFinishThreads, 4) verify_finish(VerifyKArgs a, int n_comb) {
  grid_dep_wait();
  grid_dep_launch_dependents();
  if ((int)blockIdx.x < n_comb) combine_row<D>(a, blockIdx.x);
  else finalize_chunk(a, blockIdx.x - n_comb);
}

// ---------------------------------------------------------------------------

cudaError_t launch_split_tc(const VerifyKArgs& k, const ds_verify_args& a,
                            const VerifyLayout& L, cudaStream_t stream);

template <int D>
static cudaError_t launch_d(const VerifyKArgs& k, const ds_verify_args& a,
                            const VerifyLayout& L, int batch, cudaStream_t stream,
                            cudaEvent_t ev0, cudaEvent_t ev1) {
  if (ev0) cudaEventRecord(ev0, stream);
  cudaError_t e = launch_split_tc(k, a, L, stream);
  if (e != cudaSuccess) return e;
  if (ev1) cudaEventRecord(ev1, stream);
  const int n_comb = batch * k.plan.num_kv_heads * L.rg_max * (kRowsPerGroup / kFinishWarps);
  const int n_fin = k.plan.max_chunks > 0
                        ? batch * ((k.plan.max_chunks + kFinishWarps - 1) / kFinishWarps)
                        : 0;
  return launch_dependent(verify_finish<D>, dim3(n_comb + n_fin), dim3(kFinishThreads), 0,
                          stream, k, n_comb);
}

cudaError_t launch_verify(const ds_verify_args& a, const VerifyLayout& L,
                          cudaStream_t stream) {
  VerifyKArgs k;
  unsigned char* ws = static_cast<unsigned char*>(a.workspace);
  k.q = static_cast<const __nv_bfloat16*>(a.q);
  k.k = static_cast<const __nv_bfloat16*>(a.k_cache);
  k.v = static_cast<const __nv_bfloat16*>(a.v_cache);
  k.page_table = a.page_table;
  k.parents = a.parents;
  k.plan.ctx_lens = a.ctx_lens;
  k.plan.tree_offsets = a.tree_offsets;
  k.plan.batch = a.batch;
  k.plan.n_nodes = a.n_nodes;
  k.plan.num_kv_heads = a.num_kv_heads;
  k.plan.group = L.group;
  k.plan.page_size = a.page_size;
  k.plan.max_pages = a.max_pages;
  k.plan.chunk_size = a.chunk_size;
  k.plan.max_chunks = a.max_chunks;
  k.plan.target_ctas = L.target_ctas;
  k.plan.rg_max = L.rg_max;
  k.plan.status = reinterpret_cast<uint32_t*>(ws);
  k.num_q_heads = a.num_q_heads;
  k.num_pages = a.num_pages;
  const int64_t D = a.head_dim, P = a.page_size, H = a.num_kv_heads;
  if (a.kv_layout == DS_KV_NHD) {
    k.page_stride = P * H * D; k.tok_stride = H * D; k.head_stride = D;
  } else {
    k.page_stride = H * P * D; k.tok_stride = D; k.head_stride = P * D;
  }
  const float scale = a.scale != 0.f ? a.scale : 1.0f / sqrtf((float)a.head_dim);
  k.scale_log2 = scale * kLog2e;
  k.counters = reinterpret_cast<uint32_t*>(ws + L.counters);
  k.gdesc = reinterpret_cast<int4*>(ws + L.gdesc);
  k.o_part = reinterpret_cast<float*>(ws + L.o_part);
  k.lse_part = reinterpret_cast<float*>(ws + L.lse_part);
  k.clse = reinterpret_cast<float*>(ws + L.clse);
  k.row_lse = reinterpret_cast<float*>(ws + L.row_lse);
  k.out = a.out;
  k.out_f32 = a.out_dtype == DS_OUT_F32;
  k.scores = a.chunk_scores;
  k.accumulate = a.accumulate_scores;
  cudaEvent_t ev0 = static_cast<cudaEvent_t>(a.prof_event_start);
  cudaEvent_t ev1 = static_cast<cudaEvent_t>(a.prof_event_stop);
  if (a.head_dim == 128) return launch_d<128>(k, a, L, a.batch, stream, ev0, ev1);
  return launch_d<64>(k, a, L, a.batch, stream, ev0, ev1);
}

}  // namespace ds
