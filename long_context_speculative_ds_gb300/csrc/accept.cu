// Tree acceptance: greedy accept-if-equal or exact tree rejection sampling
// (vllm.cpp docs "Speculative decoding", MTP; adaptive-specdec README,
// "Correctness first" and "The controller").
//
// Greedy
//   argmax pass (kArgmaxSlices CTAs per tree node, no cluster): each CTA
//     streams one slice of the node's target row with 16-byte loads and
//     writes the slice's largest key (order-preserving logit bits << 32 |
//     ~index), so the largest key over the slices is the row's maximum at
//     its lowest index.
// Rejection
//   node pass (one cluster of 8 CTAs per tree node, each CTA one eighth of
//     the vocabulary, partial results combined through distributed shared
//     memory).  The CTA keeps its slice of the node's residual r in shared
//     memory, so every vocabulary pass after the first reads it there:
//       target max and sum exp(l - max), and the same for the draft;
//       for the k-th child of the node the residual normaliser
//         Z_k = sum_y max(0, r_{k-1}(y) - q(y)),  r_0 = p,
//         r_k = max(0, r_{k-1} - q) / Z_k  (r_k = r_{k-1} when Z_k = 0),
//       one pass per child (r updated in place), which does not depend on
//       the children's tokens, so every node's residual chain is computed in
//       parallel before the walk;
//       the bonus token the walk would draw if it stopped here: the smallest
//       x with sum_{y<=x} r_m(y) > u * sum_y r_m(y), m = number of children.
//     A leaf needs only its target row (its draft row is never read).
//     Per-element values are fp32; sums are compensated fp32 pairs, added in
//     float64 only across the cluster's eight CTAs.  Vocabularies whose slice would not fit in
//     shared memory use a streaming variant that recomputes p, q and the
//     chain from the logits on every pass.
// walk (one warp per sequence): follows the tree from the root.  Greedy
//   compares draft tokens with the argmax; rejection evaluates p(x), q(x) and
//   the residual chain at the proposed token with the node pass's own fp32
//   operations and stored scalars, and tests u * q(x) < r(x).
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "dev_common.cuh"
#include "internal.h"
#include "pdl.cuh"

namespace cg = cooperative_groups;

namespace ds {

constexpr int kAccCluster = 8;
constexpr int kAccThreads = 512;
constexpr int kAccWarps = kAccThreads / 32;
constexpr int kArgThreads = 256;
// largest shared-memory slice (floats) of the in-shared-memory rejection pass
constexpr int kRejMaxSlice = 40 * 1024;

struct AcceptKArgs {
  int32_t mode;
  const float* tl;
  const float* dl;
  const int32_t* tokens;
  const int32_t* parents;
  const int32_t* offsets;
  const float* uniforms;
  int32_t batch, n_nodes, vocab;
  int32_t slices;      // greedy argmax slices per node
  int32_t vec;         // rows 16-byte aligned (vocab % 4 == 0, aligned bases)
  NodeStats* stats;
  int32_t* out_path;
  int32_t* out_n;
  int32_t* out_bonus;
  uint32_t* status;
};

// Kahan-compensated fp32 accumulator.
struct Kahan {
  float s = 0.f, c = 0.f;
  DS_DEV void add(float x) {
    float y = x - c;
    float t = s + y;
    c = (t - s) - y;
    s = t;
  }
  DS_DEV double value() const { return (double)s - (double)c; }
};

// Sequence owning a node: largest b with offsets[b] <= node.
DS_DEV int seq_of(const int32_t* offsets, int batch, int node) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(offsets + mid) <= node) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Children of `node` in increasing local index (thread 0 of the block).  A
// malformed tree (flagged by the walk) gets no children, so no parent read
// leaves the node arrays.  Returns the sequence's first node.
DS_DEV int find_children(const AcceptKArgs& a, int node, int32_t* children, int* nch) {
  const int b = seq_of(a.offsets, a.batch, node);
  const int n0 = __ldg(a.offsets + b);
  int T = __ldg(a.offsets + b + 1) - n0;
  if (T > DS_MAX_TREE_NODES || T < 0 || n0 < 0 || n0 + T > a.n_nodes) T = 0;
  int n = 0;
  const int i = node - n0;
  for (int c = i + 1; c < T; ++c)
    if (__ldg(a.parents + n0 + c) == i) children[n++] = c;
  *nch = n;
  return n0;
}

// Key whose unsigned order is (logit ascending, then index descending).
DS_DEV uint64_t argmax_key(float v, int idx) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)u << 32) | (uint32_t)(~(uint32_t)idx);
}
DS_DEV uint64_t u64max(uint64_t a, uint64_t b) { return a > b ? a : b; }
DS_DEV uint64_t warp_max_u64(uint64_t v) {
  for (int o = 16; o > 0; o >>= 1) v = u64max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------------------
// greedy: argmax of one slice of one node's target row
__global__ void __launch_bounds__(kArgThreads) accept_argmax(AcceptKArgs a) {
  __shared__ uint64_t s_k[kArgThreads / 32];
  grid_dep_wait();
  grid_dep_launch_dependents();
  const int S = a.slices;
  const int node = blockIdx.x / S, sl = blockIdx.x % S;
  const int V = a.vocab;
  const int per = ((V + S - 1) / S + 3) & ~3;
  const int v0 = min(V, sl * per), v1 = min(V, v0 + per);
  const float* row = a.tl + (int64_t)node * V;
  uint64_t best = 0;   // below every key of a real logit
  if (a.vec) {
    // four independent 16-byte loads in flight per thread
    constexpr int kStep = 4 * kArgThreads;
    for (int x = v0 + 4 * (int)threadIdx.x; x < v1; x += 4 * kStep) {
      float4 f[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int xx = x + u * kStep;
        f[u] = xx < v1 ? __ldg(reinterpret_cast<const float4*>(row + xx))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int xx = x + u * kStep;
        if (xx < v1) {
          best = u64max(best, argmax_key(f[u].x, xx));
          best = u64max(best, argmax_key(f[u].y, xx + 1));
          best = u64max(best, argmax_key(f[u].z, xx + 2));
          best = u64max(best, argmax_key(f[u].w, xx + 3));
        }
      }
    }
  } else {
    for (int x = v0 + (int)threadIdx.x; x < v1; x += kArgThreads)
      best = u64max(best, argmax_key(__ldg(row + x), x));
  }
  best = warp_max_u64(best);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s_k[warp] = best;
  __syncthreads();
  if (warp == 0) {
    best = lane < kArgThreads / 32 ? s_k[lane] : 0;
    best = warp_max_u64(best);
    if (lane == 0) a.stats[node].amax[sl] = best;
  }
}

// ---------------------------------------------------------------------------
// rejection: node pass with the residual slice in shared memory
//
// FP64 throughput on this part is a small fraction of FP32, so per-element
// and per-thread work stays in fp32: sums are Kahan-compensated per thread
// and combined as unevaluated pairs (hi, lo) with error-free two-sums; only
// the eight per-CTA pairs of a cluster are added in float64, by one warp,
// and the derived scalars (1 / S, 1 / Z) are formed once and broadcast.

// hi + lo, |lo| small against hi
struct F2 {
  float hi, lo;
};
DS_DEV F2 two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  return {s, (a - (s - bb)) + (b - bb)};
}
DS_DEV F2 f2_add(F2 x, F2 y) {
  const F2 t = two_sum(x.hi, y.hi);
  const float lo = t.lo + x.lo + y.lo;
  const float hi = t.hi + lo;
  return {hi, lo - (hi - t.hi)};
}
DS_DEV F2 f2_shfl_xor(F2 x, int o) {
  return {__shfl_xor_sync(0xffffffffu, x.hi, o), __shfl_xor_sync(0xffffffffu, x.lo, o)};
}
DS_DEV F2 f2_shfl_up(F2 x, int o) {
  return {__shfl_up_sync(0xffffffffu, x.hi, o), __shfl_up_sync(0xffffffffu, x.lo, o)};
}
DS_DEV F2 kahan_f2(const Kahan& k) { return {k.s, -k.c}; }
// F2 of a double (hi = nearest float, lo = the rest rounded)
DS_DEV F2 f2_of(double x) {
  const float hi = (float)x;
  return {hi, (float)(x - (double)hi)};
}
// x > y for F2 values
DS_DEV bool f2_gt(F2 x, F2 y) {
  const F2 d = f2_add(x, F2{-y.hi, -y.lo});
  return d.hi > 0.f || (d.hi == 0.f && d.lo > 0.f);
}

// Running (max, sum of exp(x - max)) of one thread, the sum compensated.
struct OnlineExp {
  float m;
  Kahan k;
  DS_DEV OnlineExp() : m(-__builtin_inff()) {}
  // adds four values: rescales when the maximum moves (rarely after the
  // first values), then adds their exponentials as one pairwise partial sum
  DS_DEV void add4(float4 x) {
    const float m4 = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
    if (m4 > m) {
      const float f = m == -CUDART_INF_F ? 0.f : expf(m - m4);
      k.s *= f;
      k.c *= f;
      m = m4;
    }
    if (m == -CUDART_INF_F) return;
    k.add((expf(x.x - m) + expf(x.y - m)) + (expf(x.z - m) + expf(x.w - m)));
  }
  DS_DEV void add1(float x) { add4(make_float4(x, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F)); }
};

struct RejShared {
  F2 part[2][2];               // cluster slots (two values), used alternately
  float pmax[2][2];            // maxima beside part (online exponential sums)
  F2 red[kAccWarps][2];
  float redm[kAccWarps][2];
  double dres[2];              // cluster results, float64
  double dpre, dmine;          // value 0: partials of the CTAs before this one,
                               // and this CTA's (see rank_split)
  double btot, bpre, bmine;    // the same for the bonus draw's weights
  float fres[4];               // scalars derived by thread 0
  F2 scan[kAccWarps + 1];
  int32_t first;
  int32_t children[DS_MAX_TREE_NODES];
  int32_t nch, n0, bonus;
};

DS_DEV F2 f2_scale(F2 x, float f) {
  const float hi = x.hi * f;
  return {hi, fmaf(x.hi, f, -hi) + x.lo * f};
}

// Warp 0, lane k holding CTA k's partial d of a cluster sum: stores this
// CTA's partial and the sum of the partials of the CTAs before it (the
// slice's offset in vocabulary order).
DS_DEV void rank_split(RejShared& sh, unsigned rank, double d) {
  const int lane = threadIdx.x & 31;
  const double mine = __shfl_sync(0xffffffffu, d, rank);
  double pre = lane < (int)rank ? d : 0.0;
  for (int o = 4; o > 0; o >>= 1) pre += __shfl_xor_sync(0xffffffffu, pre, o);
  if (lane == 0) { sh.dpre = pre; sh.dmine = mine; }
}

// Cluster reduction of two compensated sums: every thread passes its pair;
// afterwards sh.dres[0..1] (float64) hold the totals over the cluster.  One
// cluster barrier per call: the slot written alternates between calls, and
// a CTA writes a slot again only after every CTA has passed the barrier of
// the call in between.
DS_DEV void cluster_sum2(cg::cluster_group& cl, RejShared& sh, int& slot, F2 x0, F2 x1) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) {
    x0 = f2_add(x0, f2_shfl_xor(x0, o));
    x1 = f2_add(x1, f2_shfl_xor(x1, o));
  }
  if (lane == 0) { sh.red[warp][0] = x0; sh.red[warp][1] = x1; }
  __syncthreads();
  if (warp == 0) {
    F2 a0 = lane < kAccWarps ? sh.red[lane][0] : F2{0.f, 0.f};
    F2 a1 = lane < kAccWarps ? sh.red[lane][1] : F2{0.f, 0.f};
    for (int o = 8; o > 0; o >>= 1) {
      a0 = f2_add(a0, f2_shfl_xor(a0, o));
      a1 = f2_add(a1, f2_shfl_xor(a1, o));
    }
    if (lane == 0) { sh.part[slot][0] = a0; sh.part[slot][1] = a1; }
  }
  cl.sync();
  if (warp == 0) {
    double d0 = 0.0, d1 = 0.0;
    if (lane < kAccCluster) {
      const F2* o = cl.map_shared_rank(&sh.part[slot][0], lane);
      const F2 p0 = o[0], p1 = o[1];
      d0 = (double)p0.hi + (double)p0.lo;
      d1 = (double)p1.hi + (double)p1.lo;
    }
    rank_split(sh, cl.block_rank(), d0);
    for (int o = 4; o > 0; o >>= 1) {
      d0 += __shfl_xor_sync(0xffffffffu, d0, o);
      d1 += __shfl_xor_sync(0xffffffffu, d1, o);
    }
    if (lane == 0) { sh.dres[0] = d0; sh.dres[1] = d1; }
  }
  slot ^= 1;
}

// The same for two online exponential sums (max, sum of exp(x - max)):
// afterwards sh.fres[0..1] hold the maxima and sh.dres[0..1] the sums
// relative to them.
DS_DEV void cluster_online2(cg::cluster_group& cl, RejShared& sh, int& slot, float m0, F2 s0,
                            float m1, F2 s1) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto merge = [](float& m, F2& s, float om, F2 os) {
    const float nm = fmaxf(m, om);
    if (nm == -CUDART_INF_F) return;
    s = f2_add(f2_scale(s, m == nm ? 1.f : expf(m - nm)),
               f2_scale(os, om == nm ? 1.f : expf(om - nm)));
    m = nm;
  };
  for (int o = 16; o > 0; o >>= 1) {
    const float om0 = __shfl_xor_sync(0xffffffffu, m0, o);
    const float om1 = __shfl_xor_sync(0xffffffffu, m1, o);
    const F2 os0 = f2_shfl_xor(s0, o), os1 = f2_shfl_xor(s1, o);
    merge(m0, s0, om0, os0);
    merge(m1, s1, om1, os1);
  }
  if (lane == 0) {
    sh.red[warp][0] = s0; sh.red[warp][1] = s1;
    sh.redm[warp][0] = m0; sh.redm[warp][1] = m1;
  }
  __syncthreads();
  if (warp == 0) {
    float a0 = -CUDART_INF_F, a1 = -CUDART_INF_F;
    F2 b0{0.f, 0.f}, b1{0.f, 0.f};
    if (lane < kAccWarps) {
      a0 = sh.redm[lane][0]; a1 = sh.redm[lane][1];
      b0 = sh.red[lane][0]; b1 = sh.red[lane][1];
    }
    for (int o = 8; o > 0; o >>= 1) {
      const float om0 = __shfl_xor_sync(0xffffffffu, a0, o);
      const float om1 = __shfl_xor_sync(0xffffffffu, a1, o);
      const F2 os0 = f2_shfl_xor(b0, o), os1 = f2_shfl_xor(b1, o);
      merge(a0, b0, om0, os0);
      merge(a1, b1, om1, os1);
    }
    if (lane == 0) {
      sh.part[slot][0] = b0; sh.part[slot][1] = b1;
      sh.pmax[slot][0] = a0; sh.pmax[slot][1] = a1;
    }
  }
  cl.sync();
  if (warp == 0) {
    float mm0 = -CUDART_INF_F, mm1 = -CUDART_INF_F;
    F2 p0{0.f, 0.f}, p1{0.f, 0.f};
    if (lane < kAccCluster) {
      const F2* o = cl.map_shared_rank(&sh.part[slot][0], lane);
      const float* om = cl.map_shared_rank(&sh.pmax[slot][0], lane);
      p0 = o[0]; p1 = o[1];
      mm0 = om[0]; mm1 = om[1];
    }
    float M0 = mm0, M1 = mm1;
    for (int o = 4; o > 0; o >>= 1) {
      M0 = fmaxf(M0, __shfl_xor_sync(0xffffffffu, M0, o));
      M1 = fmaxf(M1, __shfl_xor_sync(0xffffffffu, M1, o));
    }
    // each CTA's sum rescaled to the cluster maximum, added in float64
    double d0 = 0.0, d1 = 0.0;
    if (lane < kAccCluster) {
      if (mm0 != -CUDART_INF_F) d0 = ((double)p0.hi + (double)p0.lo) * (double)expf(mm0 - M0);
      if (mm1 != -CUDART_INF_F) d1 = ((double)p1.hi + (double)p1.lo) * (double)expf(mm1 - M1);
    }
    rank_split(sh, cl.block_rank(), d0);
    for (int o = 4; o > 0; o >>= 1) {
      d0 += __shfl_xor_sync(0xffffffffu, d0, o);
      d1 += __shfl_xor_sync(0xffffffffu, d1, o);
    }
    if (lane == 0) {
      sh.dres[0] = d0; sh.dres[1] = d1;
      sh.fres[0] = M0; sh.fres[1] = M1;
    }
  }
  slot ^= 1;
}

// 1 / x of a positive float64 total, in fp32 arithmetic (the value is a
// scalar that node pass and walk share; it need not be correctly rounded)
DS_DEV float recip_f(double x) {
  const float hi = (float)x;
  const float lo = (float)(x - (double)hi);
  const float r = 1.0f / hi;
  return fmaf(-r * lo, r, r);
}

// One pass over this CTA's slice: f(r, d) for every token, r the slice value
// (updated in place) and d the token's draft logit (0 when need_d is
// false).  Thread t takes the 16-byte groups t, t + kAccThreads, ... (the
// same tokens in every pass), four groups at a time so that four 16-byte
// loads of the draft row are in flight per thread.  f returns the value the
// thread adds to its compensated sum; four tokens' values are added
// pairwise first.
template <class F>
DS_DEV Kahan visit(const float* __restrict__ drow, float* r_s, int n, bool vec, bool need_d,
                   F f) {
  const int tid = threadIdx.x;
  Kahan acc;
  if (vec) {
    const int n4 = n >> 2;
    const float4* d4 = reinterpret_cast<const float4*>(drow);
    float4* r4 = reinterpret_cast<float4*>(r_s);
    for (int base = tid; base < n4; base += 4 * kAccThreads) {
      float4 dv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = base + u * kAccThreads;
        dv[u] = (need_d && e < n4) ? __ldg(d4 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = base + u * kAccThreads;
        if (e < n4) {
          float4 x = r4[e];
          const float a0 = f(x.x, dv[u].x), a1 = f(x.y, dv[u].y);
          const float a2 = f(x.z, dv[u].z), a3 = f(x.w, dv[u].w);
          r4[e] = x;
          acc.add((a0 + a1) + (a2 + a3));
        }
      }
    }
  } else {
    for (int e = tid; e < n; e += kAccThreads) {
      float x = r_s[e];
      acc.add(f(x, need_d ? __ldg(drow + e) : 0.f));
      r_s[e] = x;
    }
  }
  return acc;
}

__global__ void __cluster_dims__(kAccCluster, 1, 1) __launch_bounds__(kAccThreads, 2)
accept_reject_pass(AcceptKArgs a) {
  cg::cluster_group cl = cg::this_cluster();
  __shared__ RejShared sh;
  extern __shared__ float r_s[];     // this CTA's slice: t, then r
  grid_dep_wait();
  grid_dep_launch_dependents();

  const int rank = (int)cl.block_rank();
  const int node = blockIdx.x / kAccCluster;
  const int V = a.vocab;
  const int per = ((V + kAccCluster - 1) / kAccCluster + 3) & ~3;
  const int v0 = min(V, rank * per), v1 = min(V, v0 + per);
  const int n = v1 - v0;
  const float* trow = a.tl + (int64_t)node * V + v0;
  const float* drow = a.dl + (int64_t)node * V + v0;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const bool vec = a.vec != 0;

  // ---- children of the node (warp 0, lane-parallel over candidates, in
  // order); the other warps start on the target row meanwhile
  if (warp == 0) {
    const int b = seq_of(a.offsets, a.batch, node);
    const int n0 = __ldg(a.offsets + b);
    int T = __ldg(a.offsets + b + 1) - n0;
    // a malformed tree (flagged by the walk) gets no children, so no parent
    // read leaves the node arrays
    if (T > DS_MAX_TREE_NODES || T < 0 || n0 < 0 || n0 + T > a.n_nodes) T = 0;
    const int i = node - n0;
    int cnt = 0;
    for (int c0 = 0; c0 < T; c0 += 32) {
      const int c = c0 + lane;
      const bool is = c > i && c < T && __ldg(a.parents + n0 + c) == i;
      const unsigned m = __ballot_sync(0xffffffffu, is);
      if (is) sh.children[cnt + __popc(m & ((1u << lane) - 1))] = c;
      cnt += __popc(m);
    }
    if (lane == 0) { sh.nch = cnt; sh.n0 = n0; }
  }

  // ---- pass 1: the target slice into shared memory; online (max, sum of
  // exponentials) of the target, and of the draft for an inner node
  OnlineExp ot, od;
  {
    const float4 ninf = make_float4(-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F);
    if (vec) {
      const int n4 = n >> 2;
      const float4* t4 = reinterpret_cast<const float4*>(trow);
      float4* r4 = reinterpret_cast<float4*>(r_s);
      for (int base = tid; base < n4; base += 4 * kAccThreads) {
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = base + u * kAccThreads;
          x[u] = e < n4 ? __ldg(t4 + e) : ninf;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = base + u * kAccThreads;
          if (e < n4) r4[e] = x[u];
          ot.add4(x[u]);
        }
      }
    } else {
      for (int e = tid; e < n; e += kAccThreads) {
        const float x = __ldg(trow + e);
        r_s[e] = x;
        ot.add1(x);
      }
    }
  }
  __syncthreads();                  // sh.nch, sh.children
  const int nch = sh.nch;
  const bool inner = nch > 0;       // a leaf never reads its draft row
  if (inner) {
    if (vec) {
      const int n4 = n >> 2;
      const float4* d4 = reinterpret_cast<const float4*>(drow);
      const float4 ninf = make_float4(-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F);
      for (int base = tid; base < n4; base += 4 * kAccThreads) {
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = base + u * kAccThreads;
          x[u] = e < n4 ? __ldg(d4 + e) : ninf;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) od.add4(x[u]);
      }
    } else {
      for (int e = tid; e < n; e += kAccThreads) od.add1(__ldg(drow + e));
    }
  }
  int slot = 0;
  cluster_online2(cl, sh, slot, ot.m, kahan_f2(ot.k), od.m, kahan_f2(od.k));
  if (tid == 0) {
    sh.fres[2] = recip_f(sh.dres[0]);
    sh.fres[3] = inner ? recip_f(sh.dres[1]) : 0.f;
    // a leaf draws its bonus from p, proportional to exp(t - M)
    sh.btot = sh.dres[0]; sh.bpre = sh.dpre; sh.bmine = sh.dmine;
  }
  __syncthreads();
  const float Mf = sh.fres[0], Mdf = sh.fres[1];
  const float invSt = sh.fres[2], invSd = sh.fres[3];

  // ---- residual chain, one pass per child.  The slice holds r_{k-1} (the
  // target logits before the first pass, which forms p = exp(t - M) / S);
  // the pass first applies the previous step (r_{k-1} = max(0, r_{k-2} - q)
  // / Z_{k-1}) and writes it back, then adds max(0, r_{k-1} - q) into Z_k:
  // per element the same float operations, in the same order, as the walk
  // uses to evaluate the chain at a token.
  float zinv_prev = 0.f;
  for (int k = 0; k < nch; ++k) {
    const Kahan kz = visit(drow, r_s, n, vec, true, [&](float& r, float d) {
      const float q = expf(d - Mdf) * invSd;
      if (k == 0) r = expf(r - Mf) * invSt;
      else if (zinv_prev != 0.f) r = fmaxf(0.f, r - q) * zinv_prev;
      return fmaxf(0.f, r - q);
    });
    cluster_sum2(cl, sh, slot, kahan_f2(kz), F2{0.f, 0.f});
    __syncthreads();
    if (tid == 0) {
      sh.fres[2] = sh.dres[0] > 0.0 ? recip_f(sh.dres[0]) : 0.f;
      if (rank == 0) a.stats[sh.n0 + sh.children[k]].zinv_after = sh.fres[2];
      // after the last child: the bonus weights max(0, r - q) (proportional
      // to the final residual) and their totals
      sh.btot = sh.dres[0]; sh.bpre = sh.dpre; sh.bmine = sh.dmine;
    }
    __syncthreads();
    zinv_prev = sh.fres[2];
  }

  // ---- bonus draw: the smallest x with sum_{y<=x} r_m(y) > u * sum r_m.
  // The draw is scale-invariant, so it runs on weights proportional to r_m
  // whose per-CTA totals the last reduction already gave: a leaf's
  // exp(t - M) (r_m = p), an inner node's max(0, r_{m-1} - q) (r_m with
  // Z_m > 0).  Only when Z_m = 0 (r_m = r_{m-1}, the slice itself) do the
  // totals take one more pass.
  int wmode = inner ? 1 : 0;        // 0: exp(t - M), 1: max(0, r - q), 2: r
  if (inner && zinv_prev == 0.f) {
    wmode = 2;
    const Kahan kr = visit(drow, r_s, n, vec, false, [&](float& r, float) { return r; });
    cluster_sum2(cl, sh, slot, kahan_f2(kr), F2{0.f, 0.f});
    __syncthreads();
    if (tid == 0) { sh.btot = sh.dres[0]; sh.bpre = sh.dpre; sh.bmine = sh.dmine; }
  }
  if (tid == 0) {
    const double thr = (double)__ldg(a.uniforms + 2 * (int64_t)node + 1) * sh.btot;
    const bool mine = (sh.bpre <= thr && thr < sh.bpre + sh.bmine) ||
                      (rank == kAccCluster - 1 && thr >= sh.bpre + sh.bmine);
    sh.fres[3] = mine ? 1.f : 0.f;
    sh.scan[kAccWarps] = f2_of(thr - sh.bpre);   // threshold within this slice
    sh.bonus = -1;
  }
  __syncthreads();
  if (sh.fres[3] != 0.f) {
    // rounds of 4 * kAccThreads consecutive tokens, thread t taking tokens
    // 4t .. 4t + 3 of a round (one conflict-free 16-byte read); a block-wide
    // scan of the round (compensated pairs) gives each thread its prefix;
    // the first thread whose prefix passes the threshold walks its four
    const F2 thr_rel = sh.scan[kAccWarps];
    auto weight = [&](float r, float d) -> float {
      if (wmode == 0) return expf(r - Mf);
      if (wmode == 1) return fmaxf(0.f, r - expf(d - Mdf) * invSd);
      return r;
    };
    auto round_vals = [&](int base, float (&v)[4]) {
      const int e = base + 4 * tid;
      if (vec) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f), dv = x;
        if (e < n) {
          x = reinterpret_cast<const float4*>(r_s)[e >> 2];
          if (wmode == 1) dv = __ldg(reinterpret_cast<const float4*>(drow) + (e >> 2));
        }
        v[0] = weight(x.x, dv.x); v[1] = weight(x.y, dv.y);
        v[2] = weight(x.z, dv.z); v[3] = weight(x.w, dv.w);
        if (e >= n) v[0] = v[1] = v[2] = v[3] = 0.f;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          v[q] = e + q < n ? weight(r_s[e + q], wmode == 1 ? __ldg(drow + e + q) : 0.f) : 0.f;
      }
    };
    F2 running{0.f, 0.f};
    for (int base = 0; base < n; base += 4 * kAccThreads) {
      float v[4];
      round_vals(base, v);
      const F2 own = two_sum(v[0] + v[1], v[2] + v[3]);
      F2 incl = own;
      for (int o = 1; o < 32; o <<= 1) {
        const F2 y = f2_shfl_up(incl, o);
        if (lane >= o) incl = f2_add(incl, y);
      }
      if (lane == 31) sh.scan[warp] = incl;
      if (tid == 0) sh.first = 0x7fffffff;
      __syncthreads();
      F2 wpre = running;
      for (int w = 0; w < warp; ++w) wpre = f2_add(wpre, sh.scan[w]);
      F2 round_tot = running;
      for (int w = 0; w < kAccWarps; ++w) round_tot = f2_add(round_tot, sh.scan[w]);
      const F2 incl_all = f2_add(wpre, incl);
      if (base + 4 * tid < n && f2_gt(incl_all, thr_rel)) atomicMin(&sh.first, tid);
      __syncthreads();
      const int first = sh.first;
      if (first != 0x7fffffff) {
        if (tid == first) {
          F2 run = f2_add(incl_all, F2{-own.hi, -own.lo});
          int pick = min(base + 4 * tid + 3, n - 1);
          for (int q = 0; q < 4 && base + 4 * tid + q < n; ++q) {
            run = f2_add(run, F2{v[q], 0.f});
            if (f2_gt(run, thr_rel)) { pick = base + 4 * tid + q; break; }
          }
          sh.bonus = v0 + pick;
        }
        break;
      }
      running = round_tot;
      __syncthreads();              // sh.scan reused by the next round
    }
    __syncthreads();
    if (tid == 0) {
      // rounding left the threshold past the slice: its last token
      a.stats[node].bonus_stop = sh.bonus >= 0 ? sh.bonus : (n > 0 ? v1 - 1 : V - 1);
    }
  }
  if (rank == 0 && tid == 0) {
    a.stats[node].m_t = Mf;
    a.stats[node].inv_s_t = invSt;
    a.stats[node].m_d = Mdf;
    a.stats[node].inv_s_d = invSd;
  }
  // no CTA may exit while another can still read its shared memory
  cl.sync();
}

// ---------------------------------------------------------------------------
// rejection, large vocabularies: the streaming node pass (p, q and the
// residual chain recomputed from the logits on every pass; no slice kept)

struct ClusterScratch {
  float f[4];
  int32_t i[2];
  double d[4];
};

// Block reduce of (max value, lowest index) pairs and one extra max.
DS_DEV void block_argmax(float& v, int& idx, float& v2, float* s_v, int* s_i,
                         float* s_v2) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    float ov2 = __shfl_xor_sync(0xffffffffu, v2, o);
    if (ov > v || (ov == v && oi < idx)) { v = ov; idx = oi; }
    v2 = fmaxf(v2, ov2);
  }
  if (lane == 0) { s_v[warp] = v; s_i[warp] = idx; s_v2[warp] = v2; }
  __syncthreads();
  if (warp == 0) {
    v = lane < kAccWarps ? s_v[lane] : -CUDART_INF_F;
    idx = lane < kAccWarps ? s_i[lane] : 0x7fffffff;
    v2 = lane < kAccWarps ? s_v2[lane] : -CUDART_INF_F;
    for (int o = 16; o > 0; o >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, v, o);
      int oi = __shfl_xor_sync(0xffffffffu, idx, o);
      float ov2 = __shfl_xor_sync(0xffffffffu, v2, o);
      if (ov > v || (ov == v && oi < idx)) { v = ov; idx = oi; }
      v2 = fmaxf(v2, ov2);
    }
  }
  __syncthreads();
}

DS_DEV double block_sum_d(double x, double* s_d) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  x = warp_sum_d(x);
  if (lane == 0) s_d[warp] = x;
  __syncthreads();
  double r = 0.0;
  if (warp == 0) {
    r = lane < kAccWarps ? s_d[lane] : 0.0;
    r = warp_sum_d(r);
    if (lane == 0) s_d[32] = r;
  }
  __syncthreads();
  r = s_d[32];
  __syncthreads();
  return r;
}

// Sum of one double per CTA over the cluster (every CTA gets the result).
DS_DEV double cluster_sum(cg::cluster_group& cl, ClusterScratch* mine, double x,
                          int slot) {
  if (threadIdx.x == 0) mine->d[slot] = x;
  cl.sync();
  double r = 0.0;
  for (int k = 0; k < kAccCluster; ++k)
    r += cl.map_shared_rank(mine, k)->d[slot];
  cl.sync();
  return r;
}


__global__ void __cluster_dims__(kAccCluster, 1, 1) __launch_bounds__(kAccThreads)
accept_reject_pass_stream(AcceptKArgs a) {
  cg::cluster_group cl = cg::this_cluster();
  __shared__ ClusterScratch cs;
  __shared__ float s_v[kAccWarps], s_v2[kAccWarps];
  __shared__ int s_i[kAccWarps];
  __shared__ double s_d[33];
  __shared__ double s_scan[kAccWarps + 1];
  __shared__ int32_t s_children[DS_MAX_TREE_NODES];
  __shared__ int32_t s_nch, s_bonus;

  const int rank = (int)cl.block_rank();
  const int node = blockIdx.x / kAccCluster;
  const int V = a.vocab;
  const int per = ((V + kAccCluster - 1) / kAccCluster + 3) & ~3;
  const int v0 = min(V, rank * per), v1 = min(V, v0 + per);
  const float* trow = a.tl + (int64_t)node * V;
  const bool reject = true;
  const float* drow = a.dl + (int64_t)node * V;
  const bool vec = (V & 3) == 0;

  // ---- pass 1: maxima (and the target's lowest argmax)
  float mx = -CUDART_INF_F, mxd = -CUDART_INF_F;
  int ix = 0x7fffffff;
  if (vec) {
    for (int x = v0 + 4 * threadIdx.x; x < v1; x += 4 * kAccThreads) {
      float4 t4 = __ldg(reinterpret_cast<const float4*>(trow + x));
      float tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (tv[e] > mx || (tv[e] == mx && x + e < ix)) { mx = tv[e]; ix = x + e; }
      if (reject) {
        float4 d4 = __ldg(reinterpret_cast<const float4*>(drow + x));
        mxd = fmaxf(mxd, fmaxf(fmaxf(d4.x, d4.y), fmaxf(d4.z, d4.w)));
      }
    }
  } else {
    for (int x = v0 + threadIdx.x; x < v1; x += kAccThreads) {
      float tv = __ldg(trow + x);
      if (tv > mx || (tv == mx && x < ix)) { mx = tv; ix = x; }
      if (reject) mxd = fmaxf(mxd, __ldg(drow + x));
    }
  }
  block_argmax(mx, ix, mxd, s_v, s_i, s_v2);
  if (threadIdx.x == 0) { cs.f[0] = mx; cs.i[0] = ix; cs.f[1] = mxd; }
  cl.sync();
  float M = -CUDART_INF_F, Md = -CUDART_INF_F;
  int I = 0x7fffffff;
  for (int k = 0; k < kAccCluster; ++k) {
    const ClusterScratch* o = cl.map_shared_rank(&cs, k);
    float ov = o->f[0];
    int oi = o->i[0];
    if (ov > M || (ov == M && oi < I)) { M = ov; I = oi; }
    Md = fmaxf(Md, o->f[1]);
  }
  cl.sync();
  (void)I;

  // ---- pass 2: normalisers
  Kahan kt, kd;
  for (int x = v0 + threadIdx.x; x < v1; x += kAccThreads) {
    kt.add(expf(__ldg(trow + x) - M));
    kd.add(expf(__ldg(drow + x) - Md));
  }
  const double St = cluster_sum(cl, &cs, block_sum_d(kt.value(), s_d), 0);
  const double Sd = cluster_sum(cl, &cs, block_sum_d(kd.value(), s_d), 1);
  const float invSt = (float)(1.0 / St), invSd = (float)(1.0 / Sd);

  // ---- children of this node (ascending)
  const int b = seq_of(a.offsets, a.batch, node);
  const int n0 = __ldg(a.offsets + b);
  int T = __ldg(a.offsets + b + 1) - n0;
  // a malformed tree (flagged by the walk) gets no children, so no parent
  // read leaves the node arrays
  if (T > DS_MAX_TREE_NODES || T < 0 || n0 < 0 || n0 + T > a.n_nodes) T = 0;
  if (threadIdx.x == 0) {
    int nch = 0;
    const int i = node - n0;
    for (int c = i + 1; c < T; ++c)
      if (__ldg(a.parents + n0 + c) == i) s_children[nch++] = c;
    s_nch = nch;
  }
  __syncthreads();
  const int nch = s_nch;

  // ---- residual normalisers, one pass per child
  float zinv[DS_MAX_TREE_NODES];  // only the first k entries are read
  float zpos[DS_MAX_TREE_NODES];
  for (int k = 0; k < nch; ++k) {
    Kahan kz;
    for (int x = v0 + threadIdx.x; x < v1; x += kAccThreads) {
      const float p = expf(__ldg(trow + x) - M) * invSt;
      const float q = expf(__ldg(drow + x) - Md) * invSd;
      float r = p;
      for (int j = 0; j < k; ++j)
        if (zpos[j] > 0.f) r = fmaxf(0.f, r - q) * zinv[j];
      kz.add(fmaxf(0.f, r - q));
    }
    const double Z = cluster_sum(cl, &cs, block_sum_d(kz.value(), s_d), 2);
    zpos[k] = Z > 0.0 ? 1.f : 0.f;
    zinv[k] = Z > 0.0 ? (float)(1.0 / Z) : 0.f;
    if (rank == 0 && threadIdx.x == 0) a.stats[n0 + s_children[k]].zinv_after = zinv[k];
  }

  // ---- bonus if the walk stops here: inverse CDF of r_nch
  auto rval = [&](int x) -> float {
    const float p = expf(__ldg(trow + x) - M) * invSt;
    const float q = expf(__ldg(drow + x) - Md) * invSd;
    float r = p;
    for (int j = 0; j < nch; ++j)
      if (zpos[j] > 0.f) r = fmaxf(0.f, r - q) * zinv[j];
    return r;
  };
  Kahan ks;
  for (int x = v0 + threadIdx.x; x < v1; x += kAccThreads) ks.add(rval(x));
  const double my_tot = block_sum_d(ks.value(), s_d);
  if (threadIdx.x == 0) cs.d[3] = my_tot;
  cl.sync();
  double pre = 0.0, tot = 0.0;
  for (int k = 0; k < kAccCluster; ++k) {
    double t = cl.map_shared_rank(&cs, k)->d[3];
    if (k < rank) pre += t;
    tot += t;
  }
  cl.sync();
  const double u = (double)__ldg(a.uniforms + 2 * (int64_t)node + 1);
  const double thr = u * tot;
  const bool mine = (pre <= thr && thr < pre + my_tot) ||
                    (rank == kAccCluster - 1 && thr >= pre + my_tot);
  if (mine) {
    // scan the slice in rounds of kAccThreads x 4 consecutive tokens
    if (threadIdx.x == 0) s_bonus = -1;
    __syncthreads();
    double running = pre;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int base = v0; base < v1; base += 4 * kAccThreads) {
      const int x0 = base + 4 * threadIdx.x;
      float e[4];
      double ts = 0.0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        e[q] = (x0 + q < v1) ? rval(x0 + q) : 0.f;
        ts += (double)e[q];
      }
      // block inclusive scan of ts
      double incl = ts;
      for (int o = 1; o < 32; o <<= 1) {
        double t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (lane == 31) s_scan[warp] = incl;
      __syncthreads();
      if (warp == 0) {
        double w = lane < kAccWarps ? s_scan[lane] : 0.0;
        double wi = w;
        for (int o = 1; o < 32; o <<= 1) {
          double t = __shfl_up_sync(0xffffffffu, wi, o);
          if (lane >= o) wi += t;
        }
        if (lane < kAccWarps) s_scan[lane] = wi - w;
        if (lane == kAccWarps - 1) s_scan[kAccWarps] = wi;
      }
      __syncthreads();
      const double excl = running + s_scan[warp] + incl - ts;
      const double round_tot = s_scan[kAccWarps];
      const bool over = excl + ts > thr && x0 < v1;
      // first thread (lowest x0) whose inclusive prefix exceeds thr
      unsigned m = __ballot_sync(0xffffffffu, over);
      if (lane == 0) s_v[warp] = m ? (float)(warp * 32 + __ffs(m) - 1) : -1.f;
      __syncthreads();
      int first = -1;
      for (int w = 0; w < kAccWarps; ++w)
        if (s_v[w] >= 0.f) { first = (int)s_v[w]; break; }
      if (first >= 0) {
        if ((int)threadIdx.x == first) {
          double run = excl;
          int pick = -1;
          for (int q = 0; q < 4 && x0 + q < v1; ++q) {
            run += (double)e[q];
            if (run > thr) { pick = x0 + q; break; }
          }
          if (pick < 0) pick = min(x0 + 3, v1 - 1);
          s_bonus = pick;
        }
        __syncthreads();
        break;
      }
      running += round_tot;
      __syncthreads();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int pick = s_bonus;
      if (pick < 0) pick = V - 1;  // rounding left the threshold past the end
      a.stats[node].bonus_stop = pick;
    }
  }
  if (rank == 0 && threadIdx.x == 0) {
    a.stats[node].m_t = M;
    a.stats[node].inv_s_t = invSt;
    a.stats[node].m_d = Md;
    a.stats[node].inv_s_d = invSd;
  }
  cl.sync();
}


// ---------------------------------------------------------------------------
// walk

// Target argmax of a node from its slices' keys (the whole warp calls it).
DS_DEV int greedy_argmax(const AcceptKArgs& a, int node) {
  const int lane = threadIdx.x & 31;
  uint64_t k = lane < a.slices ? a.stats[node].amax[lane] : 0;
  k = warp_max_u64(k);
  return (int)(~(uint32_t)(k & 0xffffffffu));
}

// One warp per sequence.
__global__ void __launch_bounds__(128) accept_walk(AcceptKArgs a) {
  grid_dep_wait();
  grid_dep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (b >= a.batch) return;
  const int n0 = __ldg(a.offsets + b), n1 = __ldg(a.offsets + b + 1);
  int T = n1 - n0;
  int32_t* path = a.out_path + (int64_t)b * DS_MAX_TREE_NODES;
  path[lane] = -1;
  path[lane + 32] = -1;
  if (T < 0 || T > DS_MAX_TREE_NODES || n0 < 0 || n1 > a.n_nodes) {
    if (lane == 0) flag(a.status, DS_DEV_BAD_TREE);
    T = 0;
  }
  if (T == 0) {
    if (lane == 0) { a.out_n[b] = 0; a.out_bonus[b] = -1; }
    return;
  }
  const bool reject = a.mode == DS_ACCEPT_REJECT;
  const int V = a.vocab;
  int i = 0, n = 0;
  for (int step = 0; step < DS_MAX_TREE_NODES; ++step) {
    const int c0 = lane, c1 = lane + 32;
    const bool k0 = c0 > i && c0 < T && __ldg(a.parents + n0 + c0) == i;
    const bool k1 = c1 > i && c1 < T && __ldg(a.parents + n0 + c1) == i;
    int next = -1;
    if (!reject) {
      const int y = greedy_argmax(a, n0 + i);
      const bool m0 = k0 && __ldg(a.tokens + n0 + c0) == y;
      const bool m1 = k1 && __ldg(a.tokens + n0 + c1) == y;
      const unsigned b0 = __ballot_sync(0xffffffffu, m0);
      const unsigned b1 = __ballot_sync(0xffffffffu, m1);
      next = b0 ? __ffs(b0) - 1 : (b1 ? 32 + __ffs(b1) - 1 : -1);
    } else {
      const uint64_t kids = (uint64_t)__ballot_sync(0xffffffffu, k0) |
                            ((uint64_t)__ballot_sync(0xffffffffu, k1) << 32);
      if (lane == 0) {
        const NodeStats st = a.stats[n0 + i];
        uint64_t rest = kids;
        uint64_t rejected = 0;
        while (rest) {
          const int c = __ffsll((long long)rest) - 1;
          rest &= rest - 1;
          const int x = __ldg(a.tokens + n0 + c);
          if (x < 0 || x >= V) {
            flag(a.status, DS_DEV_BAD_TOKEN);
            rejected |= 1ull << c;
            continue;
          }
          // p(x), q(x) and the residual after the rejected siblings, with
          // the node pass's own float operations and scalars
          const float p =
              expf(__ldg(a.tl + (int64_t)(n0 + i) * V + x) - st.m_t) * st.inv_s_t;
          const float q =
              expf(__ldg(a.dl + (int64_t)(n0 + i) * V + x) - st.m_d) * st.inv_s_d;
          float r = p;
          uint64_t rj = rejected;
          while (rj) {
            const int cj = __ffsll((long long)rj) - 1;
            rj &= rj - 1;
            const float zinv = a.stats[n0 + cj].zinv_after;
            if (zinv != 0.f) r = fmaxf(0.f, r - q) * zinv;
          }
          const float u = __ldg(a.uniforms + 2 * (int64_t)(n0 + c));
          if (u * q < r) { next = c; break; }
          rejected |= 1ull << c;
        }
      }
      next = __shfl_sync(0xffffffffu, next, 0);
    }
    if (next < 0) break;
    if (lane == 0) path[n] = next;
    ++n;
    i = next;
  }
  const int bonus = reject ? a.stats[n0 + i].bonus_stop : greedy_argmax(a, n0 + i);
  if (lane == 0) {
    a.out_n[b] = n;
    a.out_bonus[b] = bonus;
  }
}

cudaError_t launch_accept(const ds_accept_args& g, const AcceptLayout& L,
                          cudaStream_t stream) {
  AcceptKArgs a;
  a.mode = g.mode;
  a.tl = g.target_logits;
  a.dl = g.draft_logits;
  a.tokens = g.draft_tokens;
  a.parents = g.parents;
  a.offsets = g.tree_offsets;
  a.uniforms = g.uniforms;
  a.batch = g.batch;
  a.n_nodes = g.n_nodes;
  a.vocab = g.vocab;
  a.slices = accept_argmax_slices(g.vocab);
  const bool aligned = (reinterpret_cast<uintptr_t>(g.target_logits) & 15u) == 0 &&
                       (g.mode != DS_ACCEPT_REJECT ||
                        (reinterpret_cast<uintptr_t>(g.draft_logits) & 15u) == 0);
  a.vec = (g.vocab % 4 == 0 && aligned) ? 1 : 0;
  unsigned char* ws = static_cast<unsigned char*>(g.workspace);
  a.stats = reinterpret_cast<NodeStats*>(ws + L.node_stats);
  a.out_path = g.out_path;
  a.out_n = g.out_n_accepted;
  a.out_bonus = g.out_bonus;
  a.status = reinterpret_cast<uint32_t*>(ws);
  cudaError_t e = cudaSuccess;
  if (g.n_nodes > 0) {
    if (g.mode != DS_ACCEPT_REJECT) {
      e = launch_dependent(accept_argmax, dim3(g.n_nodes * a.slices), dim3(kArgThreads), 0,
                           stream, a);
    } else {
      const int per = ((g.vocab + kAccCluster - 1) / kAccCluster + 3) & ~3;
      if (per <= kRejMaxSlice) {
        const size_t smem = (size_t)per * sizeof(float);
        static int attr_set = 0;   // the attribute is per device function
        if (!attr_set) {
          e = cudaFuncSetAttribute(accept_reject_pass,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)(kRejMaxSlice * sizeof(float)));
          if (e != cudaSuccess) return e;
          attr_set = 1;
        }
        e = launch_dependent(accept_reject_pass, dim3(g.n_nodes * kAccCluster),
                             dim3(kAccThreads), smem, stream, a);
      } else {
        accept_reject_pass_stream<<<g.n_nodes * kAccCluster, kAccThreads, 0, stream>>>(a);
        e = cudaGetLastError();
      }
    }
    if (e != cudaSuccess) return e;
  }
  return launch_dependent(accept_walk, dim3((g.batch + 3) / 4), dim3(128), 0, stream, a);
}

}  // namespace ds
