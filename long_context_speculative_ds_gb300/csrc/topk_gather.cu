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
#include "pdl.cuh"

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
  // frequency j of the rotation as a 64-bit fraction of a turn:
  // round(rope_base^(-2j/D) / (2 pi) * 2^64), j < D/2 (host-computed)
  unsigned long long rope_turn[64];
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

// Frequencies of the local RoPE as 64-bit fractions of a turn: the exact
// value of 2^64 * base^(-2j/D) / (2 pi), rounded once (double has 53 bits;
// the product's error stays below 2^-37 of a turn at every position below
// 2^31).
void set_rope_turns(GatherKArgs& a, float base, int head_dim) {
  for (int j = 0; j < 64; ++j) {
    a.rope_turn[j] = 0ull;
    if (base > 0.f && j < head_dim / 2) {
      const double g = std::pow((double)base, -2.0 * j / head_dim) / 6.283185307179586;
      a.rope_turn[j] = (unsigned long long)std::llround(std::ldexp(g, 64));
    }
  }
}

// Candidate keys held in registers: kSelRegs per thread, so up to
// kSelRegs * kSelThreads candidates are read from memory once; candidates
// beyond that (contexts above 16K chunks) are re-read in every round.
constexpr int kSelRegs = 4;

__global__ void __launch_bounds__(kSelThreads) topk_select(GatherKArgs a) {
  __shared__ uint32_t hist[256];
  __shared__ int s_warp[33];
  __shared__ uint32_t s_prefix, s_krem;
  grid_dep_wait();                  // the scores come from the preceding kernels
  grid_dep_launch_dependents();
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31;
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

  // this thread's candidates c = kSelRegs * threadIdx.x + j (consecutive,
  // so that the selected ids leave in order with one scan per pass)
  uint32_t key[kSelRegs];
#pragma unroll
  for (int j = 0; j < kSelRegs; ++j) {
    const int c = kSelRegs * (int)threadIdx.x + j;
    key[j] = c < n_cand ? desc_key(__ldcg(sc + c)) : 0xffffffffu;
  }
  const int n_reg = min(n_cand, kSelRegs * kSelThreads);

  uint32_t prefix = 0, krem = (uint32_t)k;
  if (k > 0 && k < n_cand) {
    // radix select of the k-th smallest key, 8 bits at a time from the top
    for (int digit = 3; digit >= 0; --digit) {
      if (threadIdx.x < 256) hist[threadIdx.x] = 0;
      __syncthreads();
      const int shift = digit * 8;
      const uint32_t hi_mask = digit == 3 ? 0u : (0xffffffffu << (shift + 8));
      auto count = [&](uint32_t kk, bool valid) {
        const bool in = valid && (kk & hi_mask) == (prefix & hi_mask);
        const uint32_t bucket = in ? (kk >> shift) & 255u : 256u;
        if (in) atomicAdd(&hist[bucket], 1u);
      };
#pragma unroll
      for (int j = 0; j < kSelRegs; ++j)
        count(key[j], kSelRegs * (int)threadIdx.x + j < n_reg);
      for (int c0 = n_reg; c0 < n_cand; c0 += kSelThreads) {
        const int c = c0 + threadIdx.x;
        count(c < n_cand ? desc_key(__ldcg(sc + c)) : 0u, c < n_cand);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        // the bucket where the running count reaches krem (warp scan of 256)
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
        }
      }
      __syncthreads();
      prefix = s_prefix; krem = s_krem;
    }
  }
  // ascending ids of the selected candidates: every key below the k-th, and
  // the first krem (by index) of the keys equal to it.  The register-held
  // candidates first (each thread's are consecutive: one scan of the ties,
  // one of the positions), then any beyond them, kSelThreads at a time.
  auto classify = [&](uint32_t kk, int& take, int& eq) {
    take = eq = 0;
    if (k >= n_cand) take = 1;
    else if (k > 0) {
      if (kk < prefix) take = 1;
      else if (kk == prefix) eq = 1;
    }
  };
  int out_pos = 0, eq_seen = 0;
  {
    int take[kSelRegs], eq[kSelRegs], n_eq = 0;
#pragma unroll
    for (int j = 0; j < kSelRegs; ++j) {
      take[j] = eq[j] = 0;
      if (kSelRegs * (int)threadIdx.x + j < n_reg) classify(key[j], take[j], eq[j]);
      n_eq += eq[j];
    }
    int eq_tot;
    int eq_rank = block_excl_scan(n_eq, s_warp, &eq_tot);
    int n_take = 0;
#pragma unroll
    for (int j = 0; j < kSelRegs; ++j) {
      if (eq[j]) {
        if ((uint32_t)eq_rank < krem) take[j] = 1;
        ++eq_rank;
      }
      n_take += take[j];
    }
    eq_seen = eq_tot;
    int take_tot;
    int pos = block_excl_scan(n_take, s_warp, &take_tot);
#pragma unroll
    for (int j = 0; j < kSelRegs; ++j)
      if (take[j]) ids[pos++] = kSelRegs * (int)threadIdx.x + j;
    out_pos = take_tot;
  }
  for (int c0 = n_reg; c0 < n_cand; c0 += kSelThreads) {
    const int c = c0 + threadIdx.x;
    int take = 0, eq = 0;
    if (c < n_cand) classify(desc_key(__ldcg(sc + c)), take, eq);
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
}

// Packed pairs of fp32 and their conversion to a bf16 pair.
DS_DEV uint64_t f2pk(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
DS_DEV uint32_t bf16x2_of(uint64_t v) {   // round each half to bf16, low in bits 0..15
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
DS_DEV uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
DS_DEV uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
DS_DEV uint64_t fneg2(uint64_t a) { return a ^ 0x8000000080000000ull; }

// One compact row: source token (page pg, offset off) of every kv head into
// compact row (b, i), K rotated to local position i when rope_base > 0 (the
// whole warp calls it; pg < 0 writes zeros).  `cs` is the warp's scratch of
// D/2 (cos, sin) pairs in shared memory.
template <int D>
DS_DEV void put_row(const GatherKArgs& a, const int b, const int i, const int pg,
                    const int off, float2* cs) {
  constexpr int VPH = D / 8;                          // 16-byte vectors per head
  constexpr int HALF = D / 2;
  constexpr int NB = HALF / 8;                        // K units (8 pairs) per head
  const int lane = threadIdx.x & 31;
  const int nvec = a.num_kv_heads * VPH;
  const int64_t drow = ((int64_t)b * a.capacity + i) * a.num_kv_heads * D;
  const int64_t srow = (int64_t)pg * a.page_stride + (int64_t)off * a.tok_stride;
  if (!(a.rope_base > 0.f)) {
    for (int e = lane; e < nvec; e += 32) {
      const int h = e / VPH, vv = e % VPH;
      uint4 kx = make_uint4(0, 0, 0, 0), vx = make_uint4(0, 0, 0, 0);
      if (pg >= 0) {
        const int64_t so = srow + (int64_t)h * a.head_stride + vv * 8;
        kx = __ldg(reinterpret_cast<const uint4*>(a.src_k + so));
        vx = __ldg(reinterpret_cast<const uint4*>(a.src_v + so));
      }
      reinterpret_cast<uint4*>(a.out_k + drow)[e] = kx;
      reinterpret_cast<uint4*>(a.out_v + drow)[e] = vx;
    }
    return;
  }

  // With RoPE, K goes in units of (kv head, block of 8 pairs (j, j + D/2)):
  // 16 bytes from each half of the head.  Per round a lane loads four of the
  // row's 16-byte V vectors and two K units together, so that the row costs
  // one memory round trip, then writes V and rotates K.
  //
  // The angle i * base^(-2j/D) (positions reach tens of thousands of
  // radians) is reduced modulo one turn exactly: with g_j the frequency as a
  // 64-bit fraction of a turn (host-computed), i * g_j wraps modulo 2^64 to
  // the angle's fraction of a turn, whose top 32 bits read as a signed
  // number give x in [-1, 1) with angle = pi x (mod 2 pi).  Then sin and cos
  // of pi x in float32 (lane l: pairs l and l + 32, shared with the warp
  // through `cs`), the pair rotated in float32 and rounded to bf16.
  const int units = a.num_kv_heads * NB;
  for (int r = 0; 128 * r < nvec; ++r) {
    uint4 vx[4], lo[2], hi[2];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = 128 * r + 32 * k + lane;
      vx[k] = make_uint4(0, 0, 0, 0);
      if (e < nvec && pg >= 0) {
        const int64_t so = srow + (int64_t)(e / VPH) * a.head_stride + (e % VPH) * 8;
        vx[k] = __ldg(reinterpret_cast<const uint4*>(a.src_v + so));
      }
    }
    int hh[2], jj[2];
    bool valid[2];
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const int u = 64 * r + 32 * w + lane;
      valid[w] = u < units;
      hh[w] = u / NB;
      jj[w] = (u % NB) * 8;
      lo[w] = hi[w] = make_uint4(0, 0, 0, 0);
      if (valid[w] && pg >= 0) {
        const int64_t so = srow + (int64_t)hh[w] * a.head_stride + jj[w];
        lo[w] = __ldg(reinterpret_cast<const uint4*>(a.src_k + so));
        hi[w] = __ldg(reinterpret_cast<const uint4*>(a.src_k + so + HALF));
      }
    }
    if (r == 0) {
      __syncwarp();                 // the warp's previous row has read `cs`
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int j = lane + 32 * q;
        if (j < HALF) {
          const unsigned long long turn = (unsigned long long)(unsigned)i * a.rope_turn[j];
          const float x = (float)(int)(turn >> 32) * 4.656612873077393e-10f;   // 2^-31
          float sn, c;
          sincospif(x, &sn, &c);
          cs[j] = make_float2(c, sn);
        }
      }
      __syncwarp();
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = 128 * r + 32 * k + lane;
      if (e < nvec) reinterpret_cast<uint4*>(a.out_v + drow)[e] = vx[k];
    }
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      if (!valid[w]) continue;
      const int j0 = jj[w];
      const uint32_t* lw = reinterpret_cast<const uint32_t*>(&lo[w]);
      const uint32_t* hw = reinterpret_cast<const uint32_t*>(&hi[w]);
      const float4* c4 = reinterpret_cast<const float4*>(cs + j0);   // pairs j0 .. j0 + 7
      uint32_t ow_lo[4], ow_hi[4];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        // pairs j0 + 2 e2 and j0 + 2 e2 + 1: (cos, sin) of both in one load
        const float4 t = c4[e2];
        const uint64_t C = f2pk(t.x, t.z), S = f2pk(t.y, t.w);
        const uint64_t X = f2pk(__uint_as_float(lw[e2] << 16), __uint_as_float(lw[e2] & 0xffff0000u));
        const uint64_t Y = f2pk(__uint_as_float(hw[e2] << 16), __uint_as_float(hw[e2] & 0xffff0000u));
        // x' = x cos - y sin, y' = x sin + y cos
        ow_lo[e2] = bf16x2_of(ffma2(X, C, fneg2(fmul2(Y, S))));
        ow_hi[e2] = bf16x2_of(ffma2(X, S, fmul2(Y, C)));
      }
      uint16_t* dk = a.out_k + drow + (int64_t)hh[w] * D + j0;
      *reinterpret_cast<uint4*>(dk) = make_uint4(ow_lo[0], ow_lo[1], ow_lo[2], ow_lo[3]);
      *reinterpret_cast<uint4*>(dk + HALF) = make_uint4(ow_hi[0], ow_hi[1], ow_hi[2], ow_hi[3]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(256) gather_rows(GatherKArgs a) {
  __shared__ __align__(16) float2 s_cs[8][D / 2];
  grid_dep_launch_dependents();
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + warp;
  if (r >= a.capacity) return;
  int L = __ldg(a.ctx_lens + b);
  if (L < 0 || (int64_t)L > (int64_t)a.max_pages * a.page_size ||
      (L + a.chunk_size - 1) / a.chunk_size > a.max_chunks)
    L = 0;
  const int ws = max(0, L - a.window);
  // the sizes topk_select writes, formed here from the context length
  const int k = min(a.top_k, ws / a.chunk_size);
  const int sel_tokens = k * a.chunk_size;
  const int n = sel_tokens + (L - ws);
  // Rows are taken from the window region first (rows top_k * C .. of the
  // full-size layout, then wrapping to 0), so the first CTAs copy the recent
  // window, which does not depend on the selection, while topk_select still
  // runs; rows of selected chunks wait for it.
  const int i = (int)(((int64_t)r + (int64_t)a.top_k * a.chunk_size) % a.capacity);
  int32_t* posrow = a.out_positions + (int64_t)b * a.capacity;
  if (i >= n) {
    if (lane == 0) posrow[i] = -1;
    return;
  }
  int t;
  if (i < sel_tokens) {
    grid_dep_wait();                // the selection comes from topk_select
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
  put_row<D>(a, b, i, pg, t % a.page_size, s_cs[warp]);
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
  set_rope_turns(a, g.rope_base, g.head_dim);
  cudaError_t e = launch_dependent(topk_select, dim3(g.batch), dim3(kSelThreads), 0, stream, a);
  if (e != cudaSuccess) return e;
  dim3 grid((g.capacity + 7) / 8, g.batch);
  if (g.head_dim == 128)
    return launch_dependent(gather_rows<128>, grid, dim3(256), 0, stream, a);
  return launch_dependent(gather_rows<64>, grid, dim3(256), 0, stream, a);
}

// ---------------------------------------------------------------------------
// compact append: between retrievals the compact cache is kept and only the
// tokens committed since are appended behind its last row (the rolling
// window grows), K rotated to the appended rows' local positions.  One CTA
// per sequence, one warp per appended token.
template <int D>
__global__ void __launch_bounds__(256) compact_append(GatherKArgs a) {
  __shared__ int s_n0, s_cnt;
  __shared__ __align__(16) float2 s_cs[8][D / 2];
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
    put_row<D>(a, b, i, pg, t % a.page_size, s_cs[warp]);
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
  set_rope_turns(a, g.rope_base, g.head_dim);
  a.from_lens = g.from_lens;
  a.to_lens = g.to_lens;
  if (g.head_dim == 128)
    compact_append<128><<<g.batch, 256, 0, stream>>>(a);
  else
    compact_append<64><<<g.batch, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ds
