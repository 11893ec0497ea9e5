// Top-k chunk selection plus recent window, gathered into a compact cache
// (vllm-diffspec README, "What DiffSpec Does", last paragraph; CGCL-codes/
// DiffSpec README, "Features": physically contiguous chunk staging).
//
// select: one CTA per sequence.  Candidates are the chunks wholly before the
//   window start ws = max(0, L - W).  Each candidate gets a 32-bit key that
//   orders scores descending; a 4-digit radix select (8 bits per digit, block
//   histograms built with warp-aggregated shared-memory atomics) finds the
//   key of the k-th candidate and how many of that key to take (ties go to
//   the lower chunk index).  A block-wide scan then writes the chosen chunk
//   ids in ascending order, which is also the order of the working set.
// gather: one warp per compact row; 16-byte vector copies of the token's
//   K and V (all kv heads) from the paged source into [B, cap, H, D].
#include <cmath>

#include <cuda_runtime.h>
#include <stdint.h>

#include "dev_common.cuh"
#include "internal.h"

namespace ds {

struct GatherKArgs {
  const float* scores;
  const int32_t* ctx_lens;
  const uint16_t* src_k;
  const uint16_t* src_v;
  const int32_t* page_table;
  int32_t batch, max_chunks, num_kv_heads, head_dim, page_size, num_pages,
      max_pages, chunk_size, top_k, window, capacity;
  int64_t page_stride, tok_stride, head_stride;
  uint16_t* out_k;
  uint16_t* out_v;
  int32_t* out_positions;
  int32_t* out_len;
  int32_t* out_chunk_ids;
  uint32_t* status;
  float rope_base;           // > 0: rotate K to its local position
  double inv_freq[64];       // rope_base^(-2j/D), j < D/2 (host-computed)
  const int32_t* from_lens;  // compact append: tokens [from, to) of each sequence
  const int32_t* to_lens;
};

constexpr int kSelThreads = 1024;

// Order-preserving map of a float to uint32 (ascending), then inverted so that
// ascending keys mean descending scores.
DS_DEV uint32_t desc_key(float x) {
  uint32_t u = __float_as_uint(x);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ~u;
}

// Block exclusive scan of one int per thread (kSelThreads threads).
DS_DEV int block_excl_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
    int wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    s_warp[lane] = wi - w;           // exclusive warp offsets
    if (lane == 31) s_warp[32] = wi;  // block total
  }
  __syncthreads();
  int r = s_warp[warp] + incl - v;
  *total = s_warp[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kSelThreads) topk_select(GatherKArgs a) {
  __shared__ uint32_t hist[256];
  __shared__ int s_warp[33];
  __shared__ uint32_t s_prefix, s_krem, s_lt;
  const int b = blockIdx.x;
  int L = __ldg(a.ctx_lens + b);
  if (L < 0 || (int64_t)L > (int64_t)a.max_pages * a.page_size ||
      (L + a.chunk_size - 1) / a.chunk_size > a.max_chunks) {
    if (threadIdx.x == 0) flag(a.status, DS_DEV_BAD_LENGTH);
    L = 0;
  }
  const int ws = max(0, L - a.window);
  const int n_cand = ws / a.chunk_size;
  const int k = min(a.top_k, n_cand);
  const float* sc = a.scores + (int64_t)b * a.max_chunks;
  int32_t* ids = a.out_chunk_ids + (int64_t)b * a.top_k;

  uint32_t prefix = 0, krem = (uint32_t)k, lt = 0;
  if (k > 0 && k < n_cand) {
    // radix select of the k-th smallest desc_key, 8 bits at a time from the top
    for (int digit = 3; digit >= 0; --digit) {
      for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      const int shift = digit * 8;
      const uint32_t hi_mask = digit == 3 ? 0u : (0xffffffffu << (shift + 8));
      for (int c = threadIdx.x; c < n_cand; c += blockDim.x) {
        uint32_t key = desc_key(__ldg(sc + c));
        if ((key & hi_mask) == (prefix & hi_mask))
          atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        // find bucket where the running count reaches krem (warp scan of 256)
        const int lane = threadIdx.x;
        uint32_t cnt[8], loc = 0;
        for (int i = 0; i < 8; ++i) { cnt[i] = hist[lane * 8 + i]; loc += cnt[i]; }
        uint32_t incl = loc;
        for (int o = 1; o < 32; o <<= 1) {
          uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        uint32_t before = incl - loc;
        int found = -1;
        uint32_t below = 0;
        if (before < krem && krem <= incl) {
          uint32_t run = before;
          for (int i = 0; i < 8; ++i) {
            if (run + cnt[i] >= krem) { found = lane * 8 + i; below = run; break; }
            run += cnt[i];
          }
        }
        unsigned m = __ballot_sync(0xffffffffu, found >= 0);
        int src = __ffs(m) - 1;
        int fb = __shfl_sync(0xffffffffu, found, src);
        uint32_t bl = __shfl_sync(0xffffffffu, below, src);
        if (lane == 0) {
          s_prefix = prefix | ((uint32_t)fb << shift);
          s_krem = krem - bl;
          s_lt = lt + bl;
        }
      }
      __syncthreads();
      prefix = s_prefix; krem = s_krem; lt = s_lt;
    }
  }
  // write ascending ids of selected candidates
  int out_pos = 0, eq_seen = 0;
  for (int c0 = 0; c0 < n_cand; c0 += blockDim.x) {
    const int c = c0 + threadIdx.x;
    int take = 0, eq = 0;
    if (c < n_cand) {
      if (k >= n_cand) {
        take = 1;
      } else if (k > 0) {
        uint32_t key = desc_key(__ldg(sc + c));
        if (key < prefix) take = 1;
        else if (key == prefix) eq = 1;
      }
    }
    int eq_tot;
    int eq_rank = block_excl_scan(eq, s_warp, &eq_tot) + eq_seen;
    if (eq && (uint32_t)eq_rank < krem) take = 1;
    eq_seen += eq_tot;
    int take_tot;
    int pos = block_excl_scan(take, s_warp, &take_tot) + out_pos;
    if (take) ids[pos] = c;
    out_pos += take_tot;
  }
  for (int i = k + threadIdx.x; i < a.top_k; i += blockDim.x) ids[i] = -1;
  if (threadIdx.x == 0) a.out_len[b] = k * a.chunk_size + (L - ws);
  (void)lt;
}

// One warp per compact row.
// One compact row: source token (page pg, offset off) of every kv head into
// compact row (b, i), K rotated to local position i when rope_base > 0 (the
// whole warp calls it; pg < 0 writes zeros).
DS_DEV void put_row(const GatherKArgs& a, const int b, const int i, const int pg,
                    const int off) {
  const int lane = threadIdx.x & 31;
  const int vec_per_head = a.head_dim / 8;            // 16-byte vectors
  const int nvec = a.num_kv_heads * vec_per_head;
  const int64_t drow = ((int64_t)b * a.capacity + i) * a.num_kv_heads * a.head_dim;
  const int64_t srow = (int64_t)pg * a.page_stride + (int64_t)off * a.tok_stride;
  const bool rope = a.rope_base > 0.f;
  for (int e = lane; e < nvec; e += 32) {
    const int h = e / vec_per_head, vv = e % vec_per_head;
    uint4 kx = make_uint4(0, 0, 0, 0), vx = make_uint4(0, 0, 0, 0);
    if (pg >= 0) {
      const int64_t so = srow + (int64_t)h * a.head_stride + vv * 8;
      if (!rope) kx = __ldg(reinterpret_cast<const uint4*>(a.src_k + so));
      vx = __ldg(reinterpret_cast<const uint4*>(a.src_v + so));
    }
    if (!rope) reinterpret_cast<uint4*>(a.out_k + drow)[e] = kx;
    reinterpret_cast<uint4*>(a.out_v + drow)[e] = vx;
  }
  if (!rope) return;

  // K rotated to local position i.  The angle i * base^(-2j/D) is formed and
  // reduced modulo 2 pi in float64 (positions reach tens of thousands of
  // radians), then its sine and cosine are taken in float32 and the pair
  // (j, j + D/2) rotated in float32 and rounded to bf16.  Lane l holds the
  // sine and cosine of pairs l and l + 32.
  const int half = a.head_dim / 2;
  float cq[2], sq[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int j = lane + 32 * q;
    cq[q] = 1.f;
    sq[q] = 0.f;
    if (j < half) {
      const double ang = (double)i * a.inv_freq[j];
      const double k = rint(ang * 0.15915494309189535);           // 1 / (2 pi)
      const float r = (float)fma(-k, 6.283185307179586, ang);      // in [-pi, pi]
      sincosf(r, &sq[q], &cq[q]);
    }
  }
  // units of (kv head, block of 8 pairs), the whole warp in step so that
  // every lane takes part in every shuffle
  const int nb = half / 8;
  const int units = a.num_kv_heads * nb;
  for (int u0 = 0; u0 < units; u0 += 32) {
    const int u = u0 + lane;
    const bool valid = u < units;
    const int h = valid ? u / nb : 0, j0 = valid ? (u % nb) * 8 : 0;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
    if (valid && pg >= 0) {
      const int64_t so = srow + (int64_t)h * a.head_stride + j0;
      lo = __ldg(reinterpret_cast<const uint4*>(a.src_k + so));
      hi = __ldg(reinterpret_cast<const uint4*>(a.src_k + so + half));
    }
    const uint32_t* lw = reinterpret_cast<const uint32_t*>(&lo);
    const uint32_t* hw = reinterpret_cast<const uint32_t*>(&hi);
    uint32_t ow_lo[4], ow_hi[4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      float xo[2], yo[2];
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int j = j0 + 2 * e2 + p;
        const float c0 = __shfl_sync(0xffffffffu, cq[0], j & 31);
        const float c1 = __shfl_sync(0xffffffffu, cq[1], j & 31);
        const float s0 = __shfl_sync(0xffffffffu, sq[0], j & 31);
        const float s1 = __shfl_sync(0xffffffffu, sq[1], j & 31);
        const float c = j < 32 ? c0 : c1, sn = j < 32 ? s0 : s1;
        const float x = __uint_as_float((p ? (lw[e2] >> 16) : (lw[e2] & 0xffffu)) << 16);
        const float y = __uint_as_float((p ? (hw[e2] >> 16) : (hw[e2] & 0xffffu)) << 16);
        xo[p] = fmaf(x, c, -y * sn);
        yo[p] = fmaf(x, sn, y * c);
      }
      ow_lo[e2] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(xo[0])) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(xo[1])) << 16);
      ow_hi[e2] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(yo[0])) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(yo[1])) << 16);
    }
    if (valid) {
      uint16_t* dk = a.out_k + drow + (int64_t)h * a.head_dim + j0;
      *reinterpret_cast<uint4*>(dk) = make_uint4(ow_lo[0], ow_lo[1], ow_lo[2], ow_lo[3]);
      *reinterpret_cast<uint4*>(dk + half) = make_uint4(ow_hi[0], ow_hi[1], ow_hi[2], ow_hi[3]);
    }
  }
}

__global__ void __launch_bounds__(256) gather_rows(GatherKArgs a) {
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 8 + warp;
  if (i >= a.capacity) return;
  int L = __ldg(a.ctx_lens + b);
  if (L < 0 || (int64_t)L > (int64_t)a.max_pages * a.page_size ||
      (L + a.chunk_size - 1) / a.chunk_size > a.max_chunks)
    L = 0;
  const int ws = max(0, L - a.window);
  const int n = __ldg(a.out_len + b);
  int32_t* posrow = a.out_positions + (int64_t)b * a.capacity;
  if (i >= n) {
    if (lane == 0) posrow[i] = -1;
    return;
  }
  const int sel_tokens = n - (L - ws);
  int t;
  if (i < sel_tokens) {
    int c = __ldg(a.out_chunk_ids + (int64_t)b * a.top_k + i / a.chunk_size);
    t = c * a.chunk_size + i % a.chunk_size;
  } else {
    t = ws + (i - sel_tokens);
  }
  if (lane == 0) posrow[i] = t;
  int pg = (t >= 0 && t < L) ? __ldg(a.page_table + (int64_t)b * a.max_pages + t / a.page_size) : -1;
  if (pg < 0 || pg >= a.num_pages) {
    if (lane == 0) flag(a.status, DS_DEV_BAD_PAGE);
    pg = -1;
  }
  put_row(a, b, i, pg, t % a.page_size);
}

cudaError_t launch_topk_gather(const ds_gather_args& g, cudaStream_t stream) {
  GatherKArgs a;
  a.scores = g.scores;
  a.ctx_lens = g.ctx_lens;
  a.src_k = static_cast<const uint16_t*>(g.src_k);
  a.src_v = static_cast<const uint16_t*>(g.src_v);
  a.page_table = g.page_table;
  a.batch = g.batch; a.max_chunks = g.max_chunks; a.num_kv_heads = g.num_kv_heads;
  a.head_dim = g.head_dim; a.page_size = g.page_size; a.num_pages = g.num_pages;
  a.max_pages = g.max_pages; a.chunk_size = g.chunk_size; a.top_k = g.top_k;
  a.window = g.window; a.capacity = g.capacity;
  const int64_t D = g.head_dim, P = g.page_size, H = g.num_kv_heads;
  if (g.kv_layout == DS_KV_NHD) {
    a.page_stride = P * H * D; a.tok_stride = H * D; a.head_stride = D;
  } else {
    a.page_stride = H * P * D; a.tok_stride = D; a.head_stride = P * D;
  }
  a.out_k = static_cast<uint16_t*>(g.out_k);
  a.out_v = static_cast<uint16_t*>(g.out_v);
  a.out_positions = g.out_positions;
  a.out_len = g.out_len;
  a.out_chunk_ids = g.out_chunk_ids;
  a.status = static_cast<uint32_t*>(g.workspace);
  a.rope_base = g.rope_base;
  for (int j = 0; j < 64; ++j)
    a.inv_freq[j] = (g.rope_base > 0.f && j < g.head_dim / 2)
                        ? std::pow((double)g.rope_base, -2.0 * j / g.head_dim)
                        : 0.0;
  topk_select<<<g.batch, kSelThreads, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 grid((g.capacity + 7) / 8, g.batch);
  gather_rows<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// compact append: between retrievals the compact cache is kept and only the
// tokens committed since are appended behind its last row (the rolling
// window grows), K rotated to the appended rows' local positions.  One CTA
// per sequence, one warp per appended token.
__global__ void __launch_bounds__(256) compact_append(GatherKArgs a) {
  __shared__ int s_n0, s_cnt;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    const int n0 = __ldg(a.out_len + b);
    const int from = __ldg(a.from_lens + b), to = __ldg(a.to_lens + b);
    int cnt = to - from;
    if (from < 0 || cnt < 0 || (int64_t)to > (int64_t)a.max_pages * a.page_size ||
        n0 < 0 || n0 > a.capacity || (int64_t)n0 + cnt > a.capacity) {
      flag(a.status, DS_DEV_BAD_LENGTH);
      cnt = 0;
    }
    s_n0 = n0;
    s_cnt = cnt;
  }
  __syncthreads();
  const int n0 = s_n0, cnt = s_cnt;
  const int from = __ldg(a.from_lens + b);
  int32_t* posrow = a.out_positions + (int64_t)b * a.capacity;
  for (int k = warp; k < cnt; k += 8) {
    const int t = from + k, i = n0 + k;
    int pg = __ldg(a.page_table + (int64_t)b * a.max_pages + t / a.page_size);
    if (pg < 0 || pg >= a.num_pages) {
      if (lane == 0) flag(a.status, DS_DEV_BAD_PAGE);
      pg = -1;
    }
    if (lane == 0) posrow[i] = t;
    put_row(a, b, i, pg, t % a.page_size);
  }
  __syncthreads();
  if (threadIdx.x == 0 && cnt > 0) a.out_len[b] = n0 + cnt;
}

cudaError_t launch_compact_append(const ds_append_args& g, cudaStream_t stream) {
  GatherKArgs a{};
  a.src_k = static_cast<const uint16_t*>(g.src_k);
  a.src_v = static_cast<const uint16_t*>(g.src_v);
  a.page_table = g.page_table;
  a.batch = g.batch;
  a.num_kv_heads = g.num_kv_heads;
  a.head_dim = g.head_dim;
  a.page_size = g.page_size;
  a.num_pages = g.num_pages;
  a.max_pages = g.max_pages;
  a.capacity = g.capacity;
  const int64_t P = g.page_size, H = g.num_kv_heads, D = g.head_dim;
  if (g.kv_layout == DS_KV_NHD) {
    a.page_stride = P * H * D; a.tok_stride = H * D; a.head_stride = D;
  } else {
    a.page_stride = H * P * D; a.tok_stride = D; a.head_stride = P * D;
  }
  a.out_k = static_cast<uint16_t*>(g.out_k);
  a.out_v = static_cast<uint16_t*>(g.out_v);
  a.out_positions = g.out_positions;
  a.out_len = g.out_len;
  a.status = static_cast<uint32_t*>(g.workspace);
  a.rope_base = g.rope_base;
  for (int j = 0; j < 64; ++j)
    a.inv_freq[j] = (g.rope_base > 0.f && j < g.head_dim / 2)
                        ? std::pow((double)g.rope_base, -2.0 * j / g.head_dim)
                        : 0.0;
  a.from_lens = g.from_lens;
  a.to_lens = g.to_lens;
  compact_append<<<g.batch, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ds
