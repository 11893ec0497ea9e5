// Tree-verify attention over a paged bf16 KV cache with fused chunk salience.
//
// Three launches per call:
//   1. split pass   (tcgen05 kernel in verify_tc.cu) one CTA per work item
//                   (sequence, kv head, row group, split of key tiles):
//                   online softmax over its key tiles, writing
//                   the split's normalised output, its row log2-sum-exp, and
//                   for every context chunk in its range the chunk's log2
//                   attention mass per row (log2 sum_{t in chunk} 2^{s_t}).
//   2. combine      log-sum-exp merge of the splits of each row -> out, and the
//                   final row log2-sum-exp.
//   3. finalize     chunk score = sum over rows of 2^{chunk mass - row lse},
//                   the mass under the full softmax denominator, summed over
//                   all query heads and nodes (vllm-diffspec README,
//                   "Architecture": chunks scored from paged target KV).
// Scores are carried in log2 units (s * scale * log2 e) throughout.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "dev_common.cuh"
#include "internal.h"
#include "verify_common.cuh"

namespace ds {

// ---------------------------------------------------------------------------
// combine: one warp per (sequence, kv head, row group, row).  The split
// log2-sum-exps are read lane-parallel; split outputs are accumulated eight
// splits at a time so that eight 16-byte loads per lane are in flight.
template <int D>
__global__ void __launch_bounds__(256) verify_combine(VerifyKArgs a) {
  __shared__ Plan s_plan;
  const int per_b = a.plan.num_kv_heads * a.plan.rg_max;
  const int b = blockIdx.x / per_b;
  const int h = (blockIdx.x / a.plan.rg_max) % a.plan.num_kv_heads;
  const int rgi = blockIdx.x % a.plan.rg_max;
  if (threadIdx.x < 32) {
    Plan p = plan_find(a.plan, b, 0);
    if (threadIdx.x == 0) s_plan = p;
  }
  __syncthreads();
  const Plan p = s_plan;
  const SeqPlan& sq = p.seq;
  if (p.b < 0 || rgi >= sq.rg) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * 8 + warp;
  const int rows_here = min(kRowsPerGroup, sq.rows - rgi * kRowsPerGroup);
  if (r >= rows_here) return;
  const int G = a.plan.group;
  const int grow = rgi * kRowsPerGroup + r;
  const int node = sq.node0 + grow / G;
  const int qh = h * G + grow % G;
  const int base = sq.item_base + (h * sq.rg + rgi) * sq.splits;
  const int ns = sq.splits;
  const float* lp = a.lse_part + (int64_t)base * kRowsPerGroup + r;

  float mx = -CUDART_INF_F;
  for (int s = lane; s < ns; s += 32) mx = fmaxf(mx, __ldg(lp + (int64_t)s * kRowsPerGroup));
  mx = warp_max(mx);
  float sum = 0.f;
  for (int s = lane; s < ns; s += 32) sum += exp2f(__ldg(lp + (int64_t)s * kRowsPerGroup) - mx);
  sum = warp_sum(sum);
  const float lse = mx + log2f(sum);

  constexpr int E = D / 32;   // floats per lane (4 or 2)
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  const float* op0 = a.o_part + ((int64_t)base * kRowsPerGroup + r) * D + lane * E;
  const int64_t sstride = (int64_t)kRowsPerGroup * D;
  for (int s0 = 0; s0 < ns; s0 += 32) {
    // weight of split s0 + lane, broadcast below
    const float wl = (s0 + lane < ns)
                         ? exp2f(__ldg(lp + (int64_t)(s0 + lane) * kRowsPerGroup) - lse) : 0.f;
    const int cnt = min(32, ns - s0);
    for (int k0 = 0; k0 < cnt; k0 += 8) {
      float x[8][E];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k0 + k < cnt) {
          const float* op = op0 + (int64_t)(s0 + k0 + k) * sstride;
          if constexpr (E == 4) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(op));
            x[k][0] = v.x; x[k][1] = v.y; x[k][2] = v.z; x[k][3] = v.w;
          } else {
            const float2 v = __ldg(reinterpret_cast<const float2*>(op));
            x[k][0] = v.x; x[k][1] = v.y;
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float w = __shfl_sync(0xffffffffu, wl, (k0 + k) & 31);
        if (k0 + k < cnt && w != 0.f) {
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] = fmaf(w, x[k][e], acc[e]);
        }
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
  if (lane == 0)
    a.row_lse[(((int64_t)b * a.plan.num_kv_heads + h) * a.plan.rg_max + rgi) * kRowsPerGroup + r] = lse;
}

// ---------------------------------------------------------------------------
// finalize: one CTA per (chunk, sequence).  Warp w sums the rows of kv heads
// / row groups w, w + 8, ...; each lane keeps eight loads of chunk mass and
// eight of row log2-sum-exp in flight.
__global__ void __launch_bounds__(256) chunk_finalize(VerifyKArgs a) {
  __shared__ float s_part[8];
  const int b = blockIdx.y;
  const int c = blockIdx.x;
  const SeqPlan sq = seq_sizes(a.plan, b, false);
  const int n_ch = (sq.L + a.plan.chunk_size - 1) / a.plan.chunk_size;
  if (c >= n_ch) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float sum = 0.f;
  const int combos = a.plan.num_kv_heads * sq.rg;
  for (int cb = warp; cb < combos; cb += 8) {
    const int h = cb / sq.rg, rgi = cb % sq.rg;
    const int rows_here = min(kRowsPerGroup, sq.rows - rgi * kRowsPerGroup);
    const int64_t hb = ((int64_t)b * a.plan.num_kv_heads + h) * a.plan.rg_max + rgi;
    const float* cl = a.clse + (hb * a.plan.max_chunks + c) * kRowsPerGroup;
    const float* rl = a.row_lse + hb * kRowsPerGroup;
    float v[8], w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int r = lane + 32 * k;
      v[k] = r < rows_here ? __ldg(cl + r) : -CUDART_INF_F;
      w[k] = r < rows_here ? __ldg(rl + r) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) sum += exp2f(v[k] - w[k]);
  }
  sum = warp_sum(sum);
  if (lane == 0) s_part[warp] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int i = 0; i < 8; ++i) t += s_part[i];
    float* dst = a.scores + (int64_t)b * a.plan.max_chunks + c;
    *dst = a.accumulate ? *dst + t : t;
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
  dim3 gc(batch * k.plan.num_kv_heads * L.rg_max, kRowsPerGroup / 8);
  verify_combine<D><<<gc, 256, 0, stream>>>(k);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (k.plan.max_chunks > 0) {
    dim3 gf(k.plan.max_chunks, batch);
    chunk_finalize<<<gf, 256, 0, stream>>>(k);
    e = cudaGetLastError();
  }
  return e;
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
