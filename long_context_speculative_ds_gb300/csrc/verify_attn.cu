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
//   round trip; then the outputs of a batch of splits (lane-parallel over
//   columns) together with their log2-sum-exps (lane-parallel over splits)
//   and the row's final log2-sum-exp; the weights 2^{lse_s - lse} are
//   broadcast from the lane that holds split s.  The split outputs are bf16
//   when the final output is (f32 otherwise), and a batch is 20 bf16 splits
//   (head_dim 128) or kCombBatch f32 splits: within 64 registers, so that
//   every CTA of the launch is resident at once, and at 128K context (19
//   splits per row group) the bf16 batch is a single round trip.
// finalize (the rest): one warp per (chunk, sequence).  Lane i covers rows
//   4i .. 4i + 3 and 128 + 4i .. 128 + 4i + 3 of every (kv head, row group)
//   with 16-byte loads of the chunk masses, kFinCombos (kv head, row group)
//   combinations per round; the rows' final log2-sum-exps, the same for
//   every chunk of the sequence, are read through L1 as each round is
//   summed.
constexpr int kCombBatch = 8;
constexpr int kFinCombos = 4;   // (kv head, row group) combinations per finalize round
constexpr int kFinishThreads = 256;
constexpr int kFinishWarps = kFinishThreads / 32;

template <int D, bool HALF>
DS_DEV void combine_row(const VerifyKArgs& a, int blk) {
  const int row_blocks = kRowsPerGroup / kFinishWarps;
  const int grp = blk / row_blocks, rblk = blk % row_blocks;
  const int per_b = a.plan.num_kv_heads * a.plan.rg_max;
  const int b = grp / per_b;
  const int h = (grp / a.plan.rg_max) % a.plan.num_kv_heads;
  const int rgi = grp % a.plan.rg_max;
  const int warp = threadIdx.x >> 5;
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
  // bf16 rows are half the registers, so with head_dim 128 twenty splits
  // (and at 64, thirty-two) arrive in one round trip
  constexpr int NB = HALF ? (D == 128 ? 20 : 32) : kCombBatch;
  combine_row_splits<D, HALF, NB>(a, gd.x, gd.y, r, lse, (int64_t)node * a.num_q_heads + qh);
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
  const float4* rl_b =
      reinterpret_cast<const float4*>(a.row_lse + (int64_t)b * combos * kRowsPerGroup);
  float4 v[kFinCombos][2];
  auto load = [&](int cb0) {
#pragma unroll
    for (int k = 0; k < kFinCombos; ++k) {
      if (cb0 + k < combos) {
        const int64_t hb = (int64_t)b * combos + cb0 + k;
        const float4* cl = reinterpret_cast<const float4*>(
            a.clse + (hb * a.plan.max_chunks + c) * kRowsPerGroup);
#pragma unroll
        for (int q = 0; q < 2; ++q) v[k][q] = __ldcg(cl + lane + 32 * q);
      }
    }
  };
  load(0);
  int rows, rg;
  {
    const SeqPlan sq = seq_sizes(a.plan, b, false);
    if (c >= (sq.L + a.plan.chunk_size - 1) / a.plan.chunk_size) return;
    rows = sq.rows;
    rg = sq.rg;
  }
  float sum = 0.f;
  for (int cb0 = 0; cb0 < combos; cb0 += kFinCombos) {
    if (cb0 > 0) load(cb0);
#pragma unroll
    for (int k = 0; k < kFinCombos; ++k) {
      const int cb = cb0 + k;
      const int rgi = cb % rg_max;
      if (cb < combos && rgi < rg) {
        // rows of this lane below the row group's end
        const int left = rows - rgi * kRowsPerGroup - 4 * lane;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          // the sequence's row log2-sum-exps are the same 8 KB for every
          // warp of the sequence: read through L1 when the masses are in
          const float4 w = __ldg(rl_b + cb * (kRowsPerGroup / 4) + lane + 32 * q);
          const int n = left - 128 * q;
          if (n > 0) sum += exp2f(v[k][q].x - w.x);
          if (n > 1) sum += exp2f(v[k][q].y - w.y);
          if (n > 2) sum += exp2f(v[k][q].z - w.z);
          if (n > 3) sum += exp2f(v[k][q].w - w.w);
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
  if ((int)blockIdx.x < n_comb) {
    // split outputs are bf16 when the final output is
    if (a.out_f32) combine_row<D, false>(a, blockIdx.x);
    else combine_row<D, true>(a, blockIdx.x);
  } else {
    finalize_chunk(a, blockIdx.x - n_comb);
  }
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
  k.plan.wave_ctas = L.wave_ctas;
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
