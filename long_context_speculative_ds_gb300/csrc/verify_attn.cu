// Tree-verify attention over a paged bf16 KV cache with fused chunk salience.
//
// Three launches per call:
//   1. split pass   one CTA per work item (sequence, kv head, row group, split
//                   of key tiles): online softmax over its key tiles, writing
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
#include <stdlib.h>

#include "dev_common.cuh"
#include "internal.h"
#include "verify_common.cuh"

namespace ds {



// ---------------------------------------------------------------------------
// split pass, CUDA-core version: one thread per query row (<= 256 rows).
template <int D>
__global__ void __launch_bounds__(256, 1) verify_split_simt(VerifyKArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __nv_bfloat16* sk = reinterpret_cast<__nv_bfloat16*>(smem);          // [128][D]
  __nv_bfloat16* sv = sk + kTileKeys * D;                               // [128][D]
  __shared__ Plan s_plan;
  __shared__ int32_t s_pages[kTileKeys / 16 * 8];

  if (threadIdx.x < 32) {
    Plan p = plan_find(a.plan, -1, blockIdx.x);
    if (threadIdx.x == 0) s_plan = p;
  }
  __syncthreads();
  const Plan p = s_plan;
  if ((int)blockIdx.x >= p.total_items || p.b < 0) return;
  const SeqPlan& sq = p.seq;
  const int G = a.plan.group;
  const int item = blockIdx.x;
  const int local = item - sq.item_base;
  const int per_h = sq.rg * sq.splits;
  const int h = local / per_h;
  const int rgi = (local % per_h) / sq.splits;
  const int split = local % sq.splits;
  const int t0 = split * p.tps;
  const int t1 = min(t0 + p.tps, sq.tiles);
  const int rows_here = min(kRowsPerGroup, sq.rows - rgi * kRowsPerGroup);
  const int r = threadIdx.x;
  const bool row_ok = r < rows_here;
  const int grow = rgi * kRowsPerGroup + r;
  const int j = grow / G;
  const int qh = h * G + grow % G;
  const int L = sq.L, T = sq.T;
  const int n_ch = (L + a.plan.chunk_size - 1) / a.plan.chunk_size;
  const int C = a.plan.chunk_size;
  const int b = p.b;

  __nv_bfloat162 q2[D / 2];
  if (row_ok) {
    const __nv_bfloat162* src = reinterpret_cast<const __nv_bfloat162*>(
        a.q + ((int64_t)(sq.node0 + j) * a.num_q_heads + qh) * D);
#pragma unroll
    for (int i = 0; i < D / 2; ++i) q2[i] = src[i];
  } else {
#pragma unroll
    for (int i = 0; i < D / 2; ++i) q2[i] = __floats2bfloat162_rn(0.f, 0.f);
  }
  uint64_t anc = 0;
  if (row_ok && t1 * kTileKeys > L)
    anc = ancestor_mask(a.parents + sq.node0, j, T, a.plan.status);

  float o[D];
#pragma unroll
  for (int d = 0; d < D; ++d) o[d] = 0.f;
  float m = -CUDART_INF_F, l = 0.f, csum = 0.f;

  const int npg_tile = kTileKeys / a.plan.page_size;
  const int32_t* ptab = a.page_table + (int64_t)b * a.plan.max_pages;
  for (int t = t0; t < t1; ++t) {
    const int slot0 = t * kTileKeys;
    if (threadIdx.x < npg_tile) {
      int pi = slot0 / a.plan.page_size + threadIdx.x;
      int pg = -1;
      if (pi * a.plan.page_size < L + T) {
        pg = __ldg(ptab + pi);
        if (pg < 0 || pg >= a.num_pages) {
          flag(a.plan.status, DS_DEV_BAD_PAGE);
          pg = -1;
        }
      }
      s_pages[threadIdx.x] = pg;
    }
    __syncthreads();
    // cooperative load of K and V tiles (16-byte vectors), zeros where invalid
    constexpr int VPR = D / 8;   // vectors per key row
    for (int e = threadIdx.x; e < kTileKeys * VPR; e += blockDim.x) {
      int kk = e / VPR, vv = e % VPR;
      int slot = slot0 + kk;
      int pg = s_pages[kk / a.plan.page_size];
      uint4 kx = make_uint4(0, 0, 0, 0), vx = make_uint4(0, 0, 0, 0);
      if (pg >= 0 && slot < L + T) {
        int64_t off = (int64_t)pg * a.page_stride +
                      (int64_t)(slot % a.plan.page_size) * a.tok_stride +
                      (int64_t)h * a.head_stride + vv * 8;
        kx = *reinterpret_cast<const uint4*>(a.k + off);
        vx = *reinterpret_cast<const uint4*>(a.v + off);
      }
      reinterpret_cast<uint4*>(sk)[kk * VPR + vv] = kx;
      reinterpret_cast<uint4*>(sv)[kk * VPR + vv] = vx;
    }
    __syncthreads();
    if (row_ok) {
      for (int sb = 0; sb < kTileKeys / 16; ++sb) {
        float s[16];
        float mloc = -CUDART_INF_F;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const int key = sb * 16 + kk;
          const int slot = slot0 + key;
          bool vis = slot < L || (slot < L + T && ((anc >> (slot - L)) & 1ull));
          const __nv_bfloat162* kr =
              reinterpret_cast<const __nv_bfloat162*>(sk + key * D);
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < D / 2; ++i) {
            float2 a2 = __bfloat1622float2(q2[i]);
            float2 b2 = __bfloat1622float2(kr[i]);
            acc = fmaf(a2.x, b2.x, acc);
            acc = fmaf(a2.y, b2.y, acc);
          }
          s[kk] = vis ? acc * a.scale_log2 : -CUDART_INF_F;
          mloc = fmaxf(mloc, s[kk]);
        }
        const float mn = fmaxf(m, mloc);
        if (mn != -CUDART_INF_F) {
          if (mn > m) {
            const float alpha = exp2f(m - mn);
            l *= alpha;
            csum *= alpha;
#pragma unroll
            for (int d = 0; d < D; ++d) o[d] *= alpha;
            m = mn;
          }
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const int key = sb * 16 + kk;
            const float pk = exp2f(s[kk] - m);
            l += pk;
            if (slot0 + key < L) csum += pk;
            const __nv_bfloat162* vr =
                reinterpret_cast<const __nv_bfloat162*>(sv + key * D);
#pragma unroll
            for (int i = 0; i < D / 2; ++i) {
              float2 v2 = __bfloat1622float2(vr[i]);
              o[2 * i] = fmaf(pk, v2.x, o[2 * i]);
              o[2 * i + 1] = fmaf(pk, v2.y, o[2 * i + 1]);
            }
          }
        }
        const int slot_end = slot0 + (sb + 1) * 16;
        if (slot_end % C == 0) {
          const int c = slot_end / C - 1;
          if (c < n_ch) {
            float val = csum > 0.f ? m + log2f(csum) : -CUDART_INF_F;
            int64_t idx = ((((int64_t)b * a.plan.num_kv_heads + h) * a.plan.rg_max + rgi) *
                               a.plan.max_chunks + c) * kRowsPerGroup + r;
            a.clse[idx] = val;
          }
          csum = 0.f;
        }
      }
    }
    __syncthreads();
  }
  if (row_ok) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float* op = a.o_part + ((int64_t)item * kRowsPerGroup + r) * D;
#pragma unroll
    for (int d = 0; d < D; d += 4)
      *reinterpret_cast<float4*>(op + d) =
          make_float4(o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv);
    a.lse_part[(int64_t)item * kRowsPerGroup + r] =
        l > 0.f ? m + log2f(l) : -CUDART_INF_F;
  }
}

// ---------------------------------------------------------------------------
// combine: one warp per (sequence, kv head, row group, row).
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

  float mx = -CUDART_INF_F;
  for (int s = lane; s < ns; s += 32)
    mx = fmaxf(mx, a.lse_part[(int64_t)(base + s) * kRowsPerGroup + r]);
  mx = warp_max(mx);
  float sum = 0.f;
  for (int s = lane; s < ns; s += 32)
    sum += exp2f(a.lse_part[(int64_t)(base + s) * kRowsPerGroup + r] - mx);
  sum = warp_sum(sum);
  const float lse = mx + log2f(sum);

  constexpr int E = D / 32;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float w = exp2f(a.lse_part[(int64_t)(base + s) * kRowsPerGroup + r] - lse);
    if (w == 0.f) continue;
    const float* op = a.o_part + ((int64_t)(base + s) * kRowsPerGroup + r) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(w, op[e], acc[e]);
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
// finalize: one warp per (sequence, chunk).
__global__ void __launch_bounds__(256) chunk_finalize(VerifyKArgs a) {
  __shared__ Plan s_plan;
  const int b = blockIdx.y;
  if (threadIdx.x < 32) {
    Plan p = plan_find(a.plan, b, 0);
    if (threadIdx.x == 0) s_plan = p;
  }
  __syncthreads();
  const Plan p = s_plan;
  if (p.b < 0) return;
  const SeqPlan& sq = p.seq;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 8 + warp;
  const int n_ch = (sq.L + a.plan.chunk_size - 1) / a.plan.chunk_size;
  if (c >= n_ch) return;
  float sum = 0.f;
  for (int h = 0; h < a.plan.num_kv_heads; ++h) {
    for (int rgi = 0; rgi < sq.rg; ++rgi) {
      const int rows_here = min(kRowsPerGroup, sq.rows - rgi * kRowsPerGroup);
      const int64_t hb = ((int64_t)b * a.plan.num_kv_heads + h) * a.plan.rg_max + rgi;
      const float* cl = a.clse + (hb * a.plan.max_chunks + c) * kRowsPerGroup;
      const float* rl = a.row_lse + hb * kRowsPerGroup;
      for (int r = lane; r < rows_here; r += 32) sum += exp2f(cl[r] - rl[r]);
    }
  }
  sum = warp_sum(sum);
  if (lane == 0) {
    float* dst = a.scores + (int64_t)b * a.plan.max_chunks + c;
    *dst = a.accumulate ? *dst + sum : sum;
  }
}

// ---------------------------------------------------------------------------

cudaError_t launch_split_tc(const VerifyKArgs& k, const ds_verify_args& a,
                            const VerifyLayout& L, cudaStream_t stream);

template <int D>
static cudaError_t launch_d(const VerifyKArgs& k, const ds_verify_args& a,
                            const VerifyLayout& L, int batch, cudaStream_t stream,
                            cudaEvent_t ev0, cudaEvent_t ev1) {
  const size_t smem = 2ull * kTileKeys * D * sizeof(__nv_bfloat16);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(verify_split_simt<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  static const bool simt = [] {
    const char* v = getenv("DS_SPLIT_IMPL");
    return v && v[0] == 's';
  }();
  if (ev0) cudaEventRecord(ev0, stream);
  cudaError_t e;
  if (simt) {
    verify_split_simt<D><<<L.max_items, 256, smem, stream>>>(k);
    e = cudaGetLastError();
  } else {
    e = launch_split_tc(k, a, L, stream);
  }
  if (e != cudaSuccess) return e;
  if (ev1) cudaEventRecord(ev1, stream);
  dim3 gc(batch * k.plan.num_kv_heads * L.rg_max, kRowsPerGroup / 8);
  verify_combine<D><<<gc, 256, 0, stream>>>(k);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 gf((k.plan.max_chunks + 7) / 8, batch);
  if (k.plan.max_chunks > 0) {
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
