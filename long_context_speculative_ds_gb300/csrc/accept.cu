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
//     the vocabulary, partial sums pushed into every CTA of the cluster
//     through distributed shared memory).  The CTA's slice of the target
//     row arrives in shared memory by one bulk copy; an inner node's draft
//     slice is loaded into registers at the same time.  Then:
//       target max and sum exp(l - max), and the same for the draft;
//       p and q of the slice, in place;
//       for the k-th child (k >= 1) the residual it is tested against, in
//         closed form r_k = max(0, p - s_k q) / C_k with s_k = 1 + C_1 +
//         ... + C_{k-1} and C_k = sum_y max(0, p - s_k q): one pass over the
//         slice and one cluster sum per child; the chain does not depend on
//         the children's tokens, so every node's chain runs in parallel
//         before the walk;
//       the bonus token the walk would draw if it stopped here: the smallest
//         x with sum_{y<=x} r_m(y) > u * sum_y r_m(y), m = number of
//         children, found by the one CTA whose slice holds the threshold.
//     A leaf needs only its target row (its draft row is never read).
//     Per-element values are fp32; sums are compensated fp32 pairs.
//     Vocabularies whose slice would not fit in registers and shared memory
//     (or rows that are not 16-byte aligned) use a streaming variant that
//     recomputes p and q from the logits on every pass.
// walk (one warp per sequence): follows the tree from the root.  Greedy
//   compares draft tokens with the argmax; rejection evaluates p(x), q(x) and
//   the proposed child's residual r(x) with the node pass's own fp32
//   operations and stored scalars, and tests u * q(x) < r(x).
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "dev_common.cuh"
#include "internal.h"
#include "pdl.cuh"
#include "tc_ptx.cuh"

namespace cg = cooperative_groups;

namespace ds {

constexpr int kAccCluster = 8;
constexpr int kAccThreads = 512;
constexpr int kAccWarps = kAccThreads / 32;
constexpr int kArgThreads = 256;

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
// rejection: node pass, target slice in shared memory, draft slice in registers
//
// FP64 throughput on this part is a small fraction of FP32, so the node pass
// computes in fp32 only: per-thread sums are Kahan-compensated and combined
// as unevaluated pairs (hi, lo) with error-free two-sums.  The eight CTAs of
// a cluster push their partial pairs into every CTA of the cluster and meet
// at one cluster barrier; every thread of every CTA then adds the same eight
// pairs in the same order, so all CTAs derive bit-identical scalars (maxima,
// 1 / S, the chain's s_k and 1 / C_k) without a broadcast.
//
// Residual chain in closed form.  With C_0 = 1, s_k = C_0 + ... + C_{k-1}
// and R_k = max(0, p - s_k q), C_k = sum_y R_k(y), the residual after k
// rejected siblings is r_k = R_k / C_k: by induction, max(0, r_{k-1} - q)
// = max(0, R_{k-1} - C_{k-1} q) / C_{k-1}, and where R_{k-1} > 0 that is
// (p - s_k q) / C_{k-1} while where R_{k-1} = 0 both sides vanish (p <= s_{k-1} q
// <= s_k q); normalising gives R_k / C_k.  So each child costs one pass of
// max(0, p - s q) over the slice and one cluster sum, never a replay of the
// earlier steps, and no per-element state changes between passes.  A zero
// residual (C_k = 0) keeps r_{k-1}, and then every later residual too.

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
DS_DEV F2 f2_shfl(F2 x, int src) {
  return {__shfl_sync(0xffffffffu, x.hi, src), __shfl_sync(0xffffffffu, x.lo, src)};
}
DS_DEV F2 kahan_f2(const Kahan& k) { return {k.s, -k.c}; }
// x * f with the product's rounding error kept
DS_DEV F2 f2_scale(F2 x, float f) {
  const float hi = x.hi * f;
  return {hi, fmaf(x.hi, f, -hi) + x.lo * f};
}
// x <= y for F2 values
DS_DEV bool f2_le(F2 x, F2 y) {
  const F2 d = f2_add(y, F2{-x.hi, -x.lo});
  return d.hi > 0.f || (d.hi == 0.f && d.lo >= 0.f);
}
DS_DEV bool f2_gt(F2 x, F2 y) { return !f2_le(x, y); }
// 1 / x of a positive pair, in fp32 (one Newton step on the pair)
DS_DEV float recip_f2(F2 x) {
  const float r = 1.0f / x.hi;
  const float e = fmaf(-x.hi, r, 1.0f) - x.lo * r;
  return fmaf(r, e, r);
}
constexpr int kRejMaxG = 10;   // 16-byte groups per thread held in registers

struct RejShared {
  uint64_t bar;                                // target slice copy
  F2 part[2][kAccCluster][2];                  // pushed CTA partials [slot][rank][value]
  float pmax[2][kAccCluster][2];               // their maxima (online sums)
  F2 red[kAccWarps][2];
  float redm[kAccWarps][2];
  float rsum[kAccWarps][kRejMaxG];             // bonus scan: warp sums per round
  F2 rtot[kRejMaxG];                           // bonus scan: round totals
  F2 wtot[kAccWarps];                          // bonus scan: warp totals of one round
  int32_t children[DS_MAX_TREE_NODES];         // local ids, in order
  int32_t ctok[DS_MAX_TREE_NODES];             // their draft tokens
  float cs[DS_MAX_TREE_NODES], cic[DS_MAX_TREE_NODES];   // their residuals (s, 1 / C)
  int32_t first, pick;
  int32_t stop, inner;                         // finish: the walk's stop node
};

// Block + cluster sum of one compensated value per thread.  Returns the
// cluster total; sh.part[slot][r][0] holds CTA r's partial afterwards (until
// the reduction after next reuses the slot).  A CTA writes slot s again only
// after every CTA has passed the barrier of the reduction in between, by
// which time every thread has finished reading slot s.
DS_DEV F2 cluster_sum(cg::cluster_group& cl, RejShared& sh, int& slot, F2 x) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned rank = cl.block_rank();
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = f2_add(x, f2_shfl_xor(x, o));
  if (lane == 0) sh.red[warp][0] = x;
  __syncthreads();
  if (warp == 0) {
    F2 y = lane < kAccWarps ? sh.red[lane][0] : F2{0.f, 0.f};
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) y = f2_add(y, f2_shfl_xor(y, o));
    y = f2_shfl(y, 0);   // one value, pushed to every CTA
    if (lane < kAccCluster) *cl.map_shared_rank(&sh.part[slot][rank][0], lane) = y;
  }
  cl.sync();
  F2 tot{0.f, 0.f};
#pragma unroll
  for (int k = 0; k < kAccCluster; ++k) tot = f2_add(tot, sh.part[slot][k][0]);
  slot ^= 1;
  return tot;
}

// The same for two online exponential sums (max, sum of exp(x - max)) per
// thread: maxima first (warp, then block), every partial rescaled once to its
// group's maximum, then compensated sums.  Returns the cluster maxima and
// sums; sh.part/pmax[slot] keep the CTA partials of value 0 for bonus_owner.
DS_DEV F2 rescale_to(F2 s, float m, float to) {
  if (m == to) return s;
  return m == -CUDART_INF_F ? F2{0.f, 0.f} : f2_scale(s, expf(m - to));
}
DS_DEV void cluster_online(cg::cluster_group& cl, RejShared& sh, int& slot, float& m0, F2& s0,
                           float& m1, F2& s1) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned rank = cl.block_rank();
  float w0 = m0, w1 = m1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    w0 = fmaxf(w0, __shfl_xor_sync(0xffffffffu, w0, o));
    w1 = fmaxf(w1, __shfl_xor_sync(0xffffffffu, w1, o));
  }
  s0 = rescale_to(s0, m0, w0);
  s1 = rescale_to(s1, m1, w1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s0 = f2_add(s0, f2_shfl_xor(s0, o));
    s1 = f2_add(s1, f2_shfl_xor(s1, o));
  }
  if (lane == 0) {
    sh.red[warp][0] = s0; sh.red[warp][1] = s1;
    sh.redm[warp][0] = w0; sh.redm[warp][1] = w1;
  }
  __syncthreads();
  if (warp == 0) {
    float a0 = -CUDART_INF_F, a1 = -CUDART_INF_F;
    F2 b0{0.f, 0.f}, b1{0.f, 0.f};
    if (lane < kAccWarps) {
      a0 = sh.redm[lane][0]; a1 = sh.redm[lane][1];
      b0 = sh.red[lane][0]; b1 = sh.red[lane][1];
    }
    float c0 = a0, c1 = a1;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      c0 = fmaxf(c0, __shfl_xor_sync(0xffffffffu, c0, o));
      c1 = fmaxf(c1, __shfl_xor_sync(0xffffffffu, c1, o));
    }
    b0 = rescale_to(b0, a0, c0);
    b1 = rescale_to(b1, a1, c1);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      b0 = f2_add(b0, f2_shfl_xor(b0, o));
      b1 = f2_add(b1, f2_shfl_xor(b1, o));
    }
    b0 = f2_shfl(b0, 0);   // one value, pushed to every CTA (the maxima are
    b1 = f2_shfl(b1, 0);   // exact, so already equal in every lane)
    if (lane < kAccCluster) {
      F2* dp = cl.map_shared_rank(&sh.part[slot][rank][0], lane);
      float* dm = cl.map_shared_rank(&sh.pmax[slot][rank][0], lane);
      dp[0] = b0; dp[1] = b1;
      dm[0] = c0; dm[1] = c1;
    }
  }
  cl.sync();
  float M0 = -CUDART_INF_F, M1 = -CUDART_INF_F;
#pragma unroll
  for (int k = 0; k < kAccCluster; ++k) {
    M0 = fmaxf(M0, sh.pmax[slot][k][0]);
    M1 = fmaxf(M1, sh.pmax[slot][k][1]);
  }
  F2 S0{0.f, 0.f}, S1{0.f, 0.f};
#pragma unroll
  for (int k = 0; k < kAccCluster; ++k) {
    S0 = f2_add(S0, rescale_to(sh.part[slot][k][0], sh.pmax[slot][k][0], M0));
    S1 = f2_add(S1, rescale_to(sh.part[slot][k][1], sh.pmax[slot][k][1], M1));
  }
  m0 = M0; s0 = S0; m1 = M1; s1 = S1;
  slot ^= 1;
}

// The CTA whose slice holds the bonus draw's threshold thr = u * total: the
// largest rank r whose prefix P_r (sum of the partials of ranks < r, added in
// rank order) is <= thr.  Every CTA evaluates the same pairs in the same
// order, so exactly one claims the draw.  `online` selects the partials of
// value 0 of an online reduction, rescaled to its maximum M.
// Returns thr - P_owner through thr_rel.
DS_DEV int bonus_owner(const RejShared& sh, int slot, bool online, float M, float u, F2& thr_rel) {
  auto part = [&](int k) {
    const F2 v = sh.part[slot][k][0];
    if (!online) return v;
    return rescale_to(v, sh.pmax[slot][k][0], M);
  };
  F2 tot{0.f, 0.f};
#pragma unroll 1
  for (int k = 0; k < kAccCluster; ++k) tot = f2_add(tot, part(k));
  const F2 thr = f2_scale(tot, u);
  F2 pre{0.f, 0.f};
  int owner = 0;
  F2 rel = thr;
#pragma unroll 1
  for (int k = 0; k < kAccCluster; ++k) {
    if (f2_le(pre, thr)) { owner = k; rel = f2_add(thr, F2{-pre.hi, -pre.lo}); }
    pre = f2_add(pre, part(k));
  }
  thr_rel = rel;
  return owner;
}

DS_DEV bool bulk_wait(uint32_t bar) {
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait(bar, 0))
    if (clock64() - t0 > (1ll << 31)) return false;
  return true;
}

// Bonus draw within one CTA's slice.  w is the node's bonus weight; thread t
// holds the 16-byte groups t + j * kAccThreads, so round j is slice tokens
// [4 * kAccThreads * j, 4 * kAccThreads * (j + 1)) in thread order.
//
// round_totals: sh.rtot[j] = compensated total of round j (warp sums, then
// pairs over the warps); returns their sum in round order, the CTA's total.
template <int G, class W>
DS_DEV F2 round_totals(RejShared& sh, int n4, W weight) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const int e = tid + j * kAccThreads;
    float v = 0.f;
    if (e < n4) {
      const float4 w = weight(j, e);
      v = (w.x + w.y) + (w.z + w.w);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sh.rsum[warp][j] = v;
  }
  if (tid == 0) { sh.first = 0x7fffffff; sh.pick = -1; }
  __syncthreads();
  if (warp < G) {
    F2 y{lane < kAccWarps ? sh.rsum[lane][warp] : 0.f, 0.f};
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) y = f2_add(y, f2_shfl_xor(y, o));
    if (lane == 0) sh.rtot[warp] = y;
  }
  __syncthreads();
  F2 tot{0.f, 0.f};
#pragma unroll
  for (int j = 0; j < G; ++j) tot = f2_add(tot, sh.rtot[j]);
  return tot;
}

// scan_round (after round_totals): the smallest slice index x with
// sum_{y <= x} w(y) > thr_rel: the round whose running total crosses the
// threshold, then a block scan of that round.  When rounding leaves the
// threshold past everything, the last token of positive weight.  Returns
// the slice index (or -1 for an empty slice).
template <int G, class W>
DS_DEV int scan_round(RejShared& sh, int n4, F2 thr_rel, W weight) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // ---- the round that crosses (every thread, the same arithmetic)
  int js = -1, jlast = -1;
  F2 base{0.f, 0.f};
  {
    F2 run{0.f, 0.f};
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const F2 rt = sh.rtot[j];
      const F2 nxt = f2_add(run, rt);
      if (js < 0 && f2_gt(nxt, thr_rel)) { js = j; base = run; }
      if (rt.hi > 0.f) jlast = j;
      run = nxt;
    }
  }
  const bool last_mode = js < 0;
  if (last_mode) js = jlast;
  if (js < 0) return n4 > 0 ? 4 * n4 - 1 : -1;   // no positive weight at all
  // ---- this thread's four weights of round js
  const int e = tid + js * kAccThreads;
  float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < G; ++j)
    if (j == js && e < n4) w = weight(j, e);
  const int x0 = 4 * e;
  if (!last_mode) {
    const F2 own = two_sum(w.x + w.y, w.z + w.w);
    F2 incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const F2 y = f2_shfl_up(incl, o);
      if (lane >= o) incl = f2_add(incl, y);
    }
    if (lane == 31) sh.wtot[warp] = incl;
    __syncthreads();
    F2 pre = base;
    for (int k = 0; k < warp; ++k) pre = f2_add(pre, sh.wtot[k]);
    const F2 incl_all = f2_add(pre, incl);
    if (e < n4 && f2_gt(incl_all, thr_rel)) atomicMin(&sh.first, tid);
    __syncthreads();
    if (tid == sh.first) {
      F2 run = f2_add(incl_all, F2{-own.hi, -own.lo});
      const float wv[4] = {w.x, w.y, w.z, w.w};
      int pick = -1;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        run = f2_add(run, F2{wv[q], 0.f});
        if (pick < 0 && f2_gt(run, thr_rel)) pick = x0 + q;
      }
      if (pick < 0) pick = x0 + 3;
      sh.pick = pick;
    }
    __syncthreads();
    if (sh.pick >= 0) return sh.pick;
  }
  // rounding left the threshold past the round: its last token of positive weight
  if (e < n4) {
    int lastpos = -1;
    if (w.x > 0.f) lastpos = x0;
    if (w.y > 0.f) lastpos = x0 + 1;
    if (w.z > 0.f) lastpos = x0 + 2;
    if (w.w > 0.f) lastpos = x0 + 3;
    if (lastpos >= 0) atomicMax(&sh.pick, lastpos);
  }
  __syncthreads();
  return sh.pick;
}

// Every CTA pushes one value (the same in all its threads) into every CTA's
// sh.part[slot][rank]; one cluster barrier.
DS_DEV void cluster_push(cg::cluster_group& cl, RejShared& sh, int& slot, F2 v) {
  if (threadIdx.x < kAccCluster)
    *cl.map_shared_rank(&sh.part[slot][cl.block_rank()][0], threadIdx.x) = v;
  cl.sync();
  slot ^= 1;
}

DS_DEV float4 expf4(float4 x, float m) {
  return make_float4(expf(x.x - m), expf(x.y - m), expf(x.z - m), expf(x.w - m));
}
DS_DEV float max4(float4 x) { return fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)); }
// max(0, p - s q) per element
DS_DEV float4 resid4(float4 p, float4 q, float s) {
  return make_float4(fmaxf(0.f, fmaf(-s, q.x, p.x)), fmaxf(0.f, fmaf(-s, q.y, p.y)),
                     fmaxf(0.f, fmaf(-s, q.z, p.z)), fmaxf(0.f, fmaf(-s, q.w, p.w)));
}
DS_DEV float sum4(float4 x) { return (x.x + x.y) + (x.z + x.w); }

// The CTA's slice of a node's rows: [v0, v1), n4 16-byte groups.
struct Slice {
  int v0, v1, n4;
};
DS_DEV Slice slice_of(int V, int rank) {
  const int per = ((V + kAccCluster - 1) / kAccCluster + 3) & ~3;
  Slice sl;
  sl.v0 = min(V, rank * per);
  sl.v1 = min(V, sl.v0 + per);
  sl.n4 = (sl.v1 - sl.v0) >> 2;
  return sl;
}

// Thread 0: the target slice of row `row` into shared memory by one bulk
// copy that completes on `bar`.
DS_DEV void copy_target_slice(const AcceptKArgs& a, int row, const Slice& sl, float4* dst,
                              uint32_t bar) {
  if (threadIdx.x != 0 || sl.n4 == 0) return;
  const uint32_t bytes = (uint32_t)sl.n4 * 16u;
  ptx::mbar_arrive_expect_tx(bar, bytes);
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(ptx::smem_addr(dst)), "l"(a.tl + (int64_t)row * a.vocab + sl.v0), "r"(bytes), "r"(bar)
      : "memory");
}

// Every thread: wait for the target slice (bounded; on a timeout the status
// records it and the copy is waited for once more before the data is used).
DS_DEV void wait_target_slice(const AcceptKArgs& a, const Slice& sl, uint32_t bar) {
  if (sl.n4 > 0 && !bulk_wait(bar)) {
    if (threadIdx.x == 0) flag(a.status, DS_DEV_TIMEOUT);
    ptx::drain_wait(bar, 0);
  }
}

// The draft slice of row `row` into registers, every load in flight at once
// (-inf outside the slice, or everywhere when `load` is false).
template <int G>
DS_DEV void load_draft_slice(const AcceptKArgs& a, int row, const Slice& sl, bool load,
                             float4 (&qv)[G]) {
  const float4* drow = reinterpret_cast<const float4*>(a.dl + (int64_t)row * a.vocab + sl.v0);
  const float4 ninf = make_float4(-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F);
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const int e = (int)threadIdx.x + j * kAccThreads;
    qv[j] = (load && e < sl.n4) ? __ldcs(drow + e) : ninf;
  }
}

// Per-thread (max, compensated sum of exp(x - max)) over the thread's groups
// of the shared slice.
template <int G>
DS_DEV void thread_online_smem(const float4* p_s, int n4, float& m, F2& s) {
  m = -CUDART_INF_F;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const int e = (int)threadIdx.x + j * kAccThreads;
    if (e < n4) m = fmaxf(m, max4(p_s[e]));
  }
  Kahan k;
  if (m != -CUDART_INF_F) {
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const int e = (int)threadIdx.x + j * kAccThreads;
      if (e < n4) k.add(sum4(expf4(p_s[e], m)));
    }
  }
  s = kahan_f2(k);
}

// One cluster of kAccCluster CTAs per tree node; CTA `rank` owns the slice
// [v0, v1) of the vocabulary, at most 4 * kAccThreads * G tokens.  Needs
// 16-byte aligned rows (vocab % 4 == 0).  A leaf leaves at once: its
// distribution matters only if the walk stops there, and then the finish
// kernel takes it.
template <int G>
__global__ void __cluster_dims__(kAccCluster, 1, 1) __launch_bounds__(kAccThreads, 2)
accept_reject_node(AcceptKArgs a) {
  cg::cluster_group cl = cg::this_cluster();
  __shared__ RejShared sh;
  extern __shared__ float4 p_s[];   // this CTA's slice: target logits, then p

  const int rank = (int)cl.block_rank();
  const int node = blockIdx.x / kAccCluster;
  const Slice sl = slice_of(a.vocab, rank);
  const int n4 = sl.n4;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t bar = ptx::smem_addr(&sh.bar);

  if (tid == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  grid_dep_wait();
  grid_dep_launch_dependents();

  // ---- children of the node, in order (every warp counts them; warp 0
  // also lists them).  A malformed tree (flagged by the walk) gets none, so
  // no parent read leaves the node arrays.
  const int b = seq_of(a.offsets, a.batch, node);
  const int n0 = __ldg(a.offsets + b);
  int nch = 0;
  {
    int T = __ldg(a.offsets + b + 1) - n0;
    if (T > DS_MAX_TREE_NODES || T < 0 || n0 < 0 || n0 + T > a.n_nodes) T = 0;
    const int i = node - n0;
    for (int c0 = 0; c0 < T; c0 += 32) {
      const int c = c0 + lane;
      const bool is = c > i && c < T && __ldg(a.parents + n0 + c) == i;
      const unsigned m = __ballot_sync(0xffffffffu, is);
      if (warp == 0 && is) {
        const int k = nch + __popc(m & ((1u << lane) - 1));
        sh.children[k] = c;
        sh.ctok[k] = __ldg(a.tokens + n0 + c);
      }
      nch += __popc(m);
    }
  }
  if (nch == 0) return;

  // ---- the target slice into shared memory, the draft slice into registers
  copy_target_slice(a, node, sl, p_s, bar);
  float4 qv[G];
  load_draft_slice<G>(a, node, sl, true, qv);
  __syncthreads();                  // the barrier's initialisation, sh.children
  wait_target_slice(a, sl, bar);

  // ---- target and draft: per thread, max m and exp(l - m), kept (target in
  // shared memory, draft in registers) with their compensated sums
  float mt = -CUDART_INF_F, md = -CUDART_INF_F;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const int e = tid + j * kAccThreads;
    if (e < n4) mt = fmaxf(mt, max4(p_s[e]));
    md = fmaxf(md, max4(qv[j]));
  }
  F2 St, Sd;
  {
    Kahan kt, kd;
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const int e = tid + j * kAccThreads;
      if (e < n4) {
        const float4 x = mt == -CUDART_INF_F ? make_float4(0.f, 0.f, 0.f, 0.f) : expf4(p_s[e], mt);
        p_s[e] = x;
        kt.add(sum4(x));
      }
      qv[j] = md == -CUDART_INF_F ? make_float4(0.f, 0.f, 0.f, 0.f) : expf4(qv[j], md);
      kd.add(sum4(qv[j]));
    }
    St = kahan_f2(kt);
    Sd = kahan_f2(kd);
  }
  float Mt = mt, Md = md;
  int slot = 0;
  cluster_online(cl, sh, slot, Mt, St, Md, Sd);
  const float invSt = recip_f2(St);
  const float invSd = recip_f2(Sd);
  NodeStats* stats = a.stats;
  if (rank == 0 && tid == 0) {
    stats[node].m_t = Mt;
    stats[node].inv_s_t = invSt;
    stats[node].m_d = Md;
    stats[node].inv_s_d = invSd;
  }
  if (tid == 0) {
    sh.cs[0] = 0.f;                  // the first child: r_0 = p
    sh.cic[0] = 1.f;
  }

  // ---- p = exp(t - m) * (exp(m - M) / S) and q likewise (each thread its
  // own groups), with the first residual's sum, max(0, p - q) (s_1 = 1)
  const float ft = mt == -CUDART_INF_F ? 0.f : expf(mt - Mt) * invSt;
  const float fd = md == -CUDART_INF_F ? 0.f : expf(md - Md) * invSd;
  Kahan k1;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const int e = tid + j * kAccThreads;
    const float4 d = qv[j];
    qv[j] = make_float4(d.x * fd, d.y * fd, d.z * fd, d.w * fd);
    if (e < n4) {
      const float4 t = p_s[e];
      const float4 pv = make_float4(t.x * ft, t.y * ft, t.z * ft, t.w * ft);
      p_s[e] = pv;
      k1.add(sum4(resid4(pv, qv[j], 1.f)));
    }
  }

  // ---- residual chain: child k (k >= 1) is tested against r_k, the
  // residual after its elder siblings were rejected; the last pass gives
  // r_nch, the bonus draw's distribution if every child is rejected
  F2 sacc{1.f, 0.f};                  // s_k = 1 + C_1 + ... + C_{k-1}
  float s_prev = 0.f, ic_prev = 1.f;  // residual in force: r_0 = p
  F2 part = kahan_f2(k1);
  for (int k = 1; k <= nch; ++k) {
    const float s = sacc.hi;
    if (k > 1) {
      Kahan kz;
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const int e = tid + j * kAccThreads;
        if (e < n4) kz.add(sum4(resid4(p_s[e], qv[j], s)));
      }
      part = kahan_f2(kz);
    }
    const F2 C = cluster_sum(cl, sh, slot, part);
    if (!(C.hi > 0.f)) {
      // zero residual: r_k = r_{k-1}, and so is every later residual
      if (tid == 0)
        for (int kk = k; kk < nch; ++kk) { sh.cs[kk] = s_prev; sh.cic[kk] = ic_prev; }
      break;
    }
    s_prev = s;
    ic_prev = recip_f2(C);
    if (k < nch && tid == 0) { sh.cs[k] = s; sh.cic[k] = ic_prev; }
    sacc = f2_add(sacc, C);
  }
  if (rank == 0 && tid == 0) stats[node].s_bonus = s_prev;

  // ---- each child's test u * q(x) < r(x), by the thread that holds its
  // token x: p(x) and q(x) are that thread's own values, so the walk needs
  // only the outcome (tokens outside the vocabulary are the walk's to flag)
  __syncthreads();                  // sh.cs, sh.cic
  for (int k = 0; k < nch; ++k) {
    const int g = sh.ctok[k] - sl.v0;
    if (g < 0 || g >= 4 * n4 || ((g >> 2) & (kAccThreads - 1)) != tid) continue;
    const int jj = (g >> 2) / kAccThreads;
    float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < G; ++j)
      if (j == jj) q4 = qv[j];
    const float4 p4 = p_s[g >> 2];
    const int c3 = g & 3;
    const float q = c3 == 0 ? q4.x : c3 == 1 ? q4.y : c3 == 2 ? q4.z : q4.w;
    const float pv = c3 == 0 ? p4.x : c3 == 1 ? p4.y : c3 == 2 ? p4.z : p4.w;
    const float r = fmaxf(0.f, fmaf(-sh.cs[k], q, pv)) * sh.cic[k];
    const int c = n0 + sh.children[k];
    stats[c].pass = __ldg(a.uniforms + 2 * (int64_t)c) * q < r ? 1 : 0;
  }
  // No CTA leaves while another can still write into its shared memory:
  // every push happens before a cluster barrier that all CTAs pass.
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

  // ---- residual chain in closed form (see the node pass above): child k
  // is tested against max(0, p - s_k q) / C_k, one pass per child
  auto pq = [&](int x, float& p, float& q) {
    p = expf(__ldg(trow + x) - M) * invSt;
    q = expf(__ldg(drow + x) - Md) * invSd;
  };
  __shared__ float s_cs[DS_MAX_TREE_NODES], s_cic[DS_MAX_TREE_NODES];
  if (threadIdx.x == 0) { s_cs[0] = 0.f; s_cic[0] = 1.f; }
  double sacc = 1.0;
  float s_prev = 0.f, s_last = 0.f;
  for (int k = 1; k <= nch; ++k) {
    const float s = (float)sacc;
    Kahan kz;
    for (int x = v0 + threadIdx.x; x < v1; x += kAccThreads) {
      float p, q;
      pq(x, p, q);
      kz.add(fmaxf(0.f, fmaf(-s, q, p)));
    }
    const double C = cluster_sum(cl, &cs, block_sum_d(kz.value(), s_d), 2);
    if (C > 0.0) {
      if (k < nch && threadIdx.x == 0) { s_cs[k] = s; s_cic[k] = (float)(1.0 / C); }
      sacc += C;
      s_prev = s;
      s_last = s;
    } else {
      // zero residual: r_k = r_{k-1}, and so is every later residual
      if (threadIdx.x == 0)
        for (int kk = k; kk < nch; ++kk) { s_cs[kk] = s_cs[k - 1]; s_cic[kk] = s_cic[k - 1]; }
      s_last = s_prev;
      break;
    }
  }

  // ---- each child's test at its token (rank 0, one thread per child)
  __syncthreads();
  if (rank == 0 && (int)threadIdx.x < nch) {
    const int k = threadIdx.x;
    const int c = n0 + s_children[k];
    const int x = __ldg(a.tokens + c);
    if (x >= 0 && x < V) {
      float p, q;
      pq(x, p, q);
      const float r = fmaxf(0.f, fmaf(-s_cs[k], q, p)) * s_cic[k];
      a.stats[c].pass = __ldg(a.uniforms + 2 * (int64_t)c) * q < r ? 1 : 0;
    }
  }

  // ---- bonus if the walk stops here: inverse CDF of the last residual
  // (p itself for a leaf)
  auto rval = [&](int x) -> float {
    float p, q;
    if (nch == 0) return expf(__ldg(trow + x) - M) * invSt;
    pq(x, p, q);
    return fmaxf(0.f, fmaf(-s_last, q, p));
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

// The walk of sequence b by one warp (every lane calls it): follows the tree
// from the root and returns the stop node (global index, -1 for an empty
// tree) and whether it has children.  With `write` it stores the path and
// the count, and the bonus -1 of an empty tree.
//
// The walk reaches child c of node i only after rejecting every elder
// sibling of c, and c's test assumes exactly that, so whether c would be
// accepted does not depend on the walk: greedy compares c's token with its
// parent's argmax, rejection reads the outcome the node pass computed; lane
// l holds nodes l and l + 32, and the walk itself is ballots over those bits.
struct WalkEnd {
  int node;
  bool inner;
};
DS_DEV WalkEnd walk_sequence(const AcceptKArgs& a, int b, bool write) {
  const int lane = threadIdx.x & 31;
  const int n0 = __ldg(a.offsets + b), n1 = __ldg(a.offsets + b + 1);
  int T = n1 - n0;
  int32_t* path = a.out_path + (int64_t)b * DS_MAX_TREE_NODES;
  if (write) {
    path[lane] = -1;
    path[lane + 32] = -1;
  }
  if (T < 0 || T > DS_MAX_TREE_NODES || n0 < 0 || n1 > a.n_nodes) {
    if (lane == 0) flag(a.status, DS_DEV_BAD_TREE);
    T = 0;
  }
  if (T == 0) {
    if (write && lane == 0) { a.out_n[b] = 0; a.out_bonus[b] = -1; }
    return {-1, false};
  }
  const bool reject = a.mode == DS_ACCEPT_REJECT;
  const int V = a.vocab;
  int par[2], tok[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = lane + 32 * h;
    par[h] = c < T ? __ldg(a.parents + n0 + c) : -1;
    tok[h] = c < T ? __ldg(a.tokens + n0 + c) : 0;
    if (!(par[h] >= 0 && par[h] < c)) par[h] = -1;   // c is a child of par[h] < c only
  }
  bool acc[2];
  if (!reject) {
    // greedy: c passes iff its token is its parent's target argmax
    int y[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = lane + 32 * h;
      uint64_t k = 0;
      if (c < T)
        for (int sl = 0; sl < a.slices; ++sl) k = u64max(k, a.stats[n0 + c].amax[sl]);
      y[h] = (int)(~(uint32_t)(k & 0xffffffffu));
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int pp = par[h] < 0 ? 0 : par[h];
      const int y0 = __shfl_sync(0xffffffffu, y[0], pp & 31);
      const int y1 = __shfl_sync(0xffffffffu, y[1], pp & 31);
      acc[h] = par[h] >= 0 && tok[h] == (pp >= 32 ? y1 : y0);
    }
  } else {
    // rejection: the node pass evaluated each child's test u * q(x) < r(x)
    // at its parent; an invalid token is flagged here and fails
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = lane + 32 * h;
      acc[h] = false;
      if (par[h] < 0) continue;
      if (tok[h] < 0 || tok[h] >= V) {
        flag(a.status, DS_DEV_BAD_TOKEN);
        continue;
      }
      acc[h] = a.stats[n0 + c].pass != 0;
    }
  }
  int i = 0, n = 0;
  bool inner = false;
  for (int step = 0; step < DS_MAX_TREE_NODES; ++step) {
    const bool k0 = par[0] == i, k1 = par[1] == i;
    const uint64_t kids = (uint64_t)__ballot_sync(0xffffffffu, k0) |
                          ((uint64_t)__ballot_sync(0xffffffffu, k1) << 32);
    const uint64_t pass = (uint64_t)__ballot_sync(0xffffffffu, k0 && acc[0]) |
                          ((uint64_t)__ballot_sync(0xffffffffu, k1 && acc[1]) << 32);
    inner = kids != 0;
    if (pass == 0) break;
    const int next = __ffsll((long long)pass) - 1;   // the first child that passes
    if (write && lane == 0) path[n] = next;
    ++n;
    i = next;
  }
  if (write && lane == 0) a.out_n[b] = n;
  return {n0 + i, inner};
}

// One warp per sequence: greedy (bonus = the stop node's argmax) and the
// streaming rejection pass (bonus drawn by the node pass).
__global__ void __launch_bounds__(128) accept_walk(AcceptKArgs a) {
  grid_dep_wait();
  grid_dep_launch_dependents();
  const int b = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (b >= a.batch) return;
  const WalkEnd w = walk_sequence(a, b, true);
  if (w.node < 0) return;
  const bool reject = a.mode == DS_ACCEPT_REJECT;
  const int bonus = reject ? a.stats[w.node].bonus_stop : greedy_argmax(a, w.node);
  if ((threadIdx.x & 31) == 0) a.out_bonus[b] = bonus;
}

// Rejection finish: one cluster per sequence.  Warp 0 of every CTA runs the
// same walk (CTA 0 writes the path); then the cluster draws the bonus token
// at the stop node: the smallest x with sum_{y<=x} w(y) > u * sum_y w(y),
// w = max(0, p - s_bonus q) after rejected children, w = exp(t - max) (that
// is, p) at a leaf, whose normaliser this kernel computes.
template <int G>
__global__ void __cluster_dims__(kAccCluster, 1, 1) __launch_bounds__(kAccThreads, 2)
accept_finish(AcceptKArgs a) {
  cg::cluster_group cl = cg::this_cluster();
  __shared__ RejShared sh;
  extern __shared__ float4 p_s[];   // the stop node's target slice
  const int rank = (int)cl.block_rank();
  const int b = blockIdx.x / kAccCluster;
  const Slice sl = slice_of(a.vocab, rank);
  const int tid = threadIdx.x;
  const uint32_t bar = ptx::smem_addr(&sh.bar);
  if (tid == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  grid_dep_wait();
  grid_dep_launch_dependents();
  if (tid < 32) {
    const WalkEnd w = walk_sequence(a, b, rank == 0);
    if (tid == 0) { sh.stop = w.node; sh.inner = w.inner ? 1 : 0; }
  }
  __syncthreads();                  // also the barrier's initialisation
  const int node = sh.stop;
  if (node < 0) return;             // empty tree (uniform over the cluster)
  const bool inner = sh.inner != 0;

  copy_target_slice(a, node, sl, p_s, bar);
  float4 wv[G];
  load_draft_slice<G>(a, node, sl, inner, wv);
  wait_target_slice(a, sl, bar);
  const float u = __ldg(a.uniforms + 2 * (int64_t)node + 1);
  int slot = 0;
  F2 thr_rel;
  int owner;
  float Mt = 0.f;
  if (inner) {
    const NodeStats st = a.stats[node];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const int e = tid + j * kAccThreads;
      float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < sl.n4) {
        const float4 t = expf4(p_s[e], st.m_t);
        const float4 d = expf4(wv[j], st.m_d);
        w = resid4(make_float4(t.x * st.inv_s_t, t.y * st.inv_s_t, t.z * st.inv_s_t,
                               t.w * st.inv_s_t),
                   make_float4(d.x * st.inv_s_d, d.y * st.inv_s_d, d.z * st.inv_s_d,
                               d.w * st.inv_s_d),
                   st.s_bonus);
      }
      wv[j] = w;
    }
    // every CTA's round totals; the CTA partials are their sums, so the
    // owner's scan sees exactly the totals the ownership was decided on
    const F2 mine = round_totals<G>(sh, sl.n4, [&](int j, int) { return wv[j]; });
    cluster_push(cl, sh, slot, mine);
    owner = bonus_owner(sh, 0, false, 0.f, u, thr_rel);
    if (owner != rank) return;
    const int x = scan_round<G>(sh, sl.n4, thr_rel, [&](int j, int) { return wv[j]; });
    if (tid == 0) a.out_bonus[b] = x >= 0 ? sl.v0 + x : a.vocab - 1;
    return;
  } else {
    F2 St, Sd{0.f, 0.f};
    float Md = -CUDART_INF_F;
    thread_online_smem<G>(p_s, sl.n4, Mt, St);
    cluster_online(cl, sh, slot, Mt, St, Md, Sd);
    owner = bonus_owner(sh, 0, true, Mt, u, thr_rel);
  }
  if (owner != rank) return;
  auto leaf_w = [&](int, int e) { return expf4(p_s[e], Mt); };
  round_totals<G>(sh, sl.n4, leaf_w);
  const int x = scan_round<G>(sh, sl.n4, thr_rel, leaf_w);
  if (tid == 0) a.out_bonus[b] = x >= 0 ? sl.v0 + x : a.vocab - 1;
  // No CTA leaves while another can still write into its shared memory:
  // every push happens before a cluster barrier that all CTAs pass.
}

template <int G>
cudaError_t launch_reject_g(const AcceptKArgs& a, int per, cudaStream_t stream) {
  static bool attr_set = false;   // the attribute is per device function
  const int max_smem = G * kAccThreads * (int)sizeof(float4);
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(accept_reject_node<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(accept_finish<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               max_smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const size_t smem = (size_t)per * sizeof(float);
  cudaError_t e = launch_dependent(accept_reject_node<G>, dim3(a.n_nodes * kAccCluster),
                                   dim3(kAccThreads), smem, stream, a);
  if (e != cudaSuccess) return e;
  return launch_dependent(accept_finish<G>, dim3(a.batch * kAccCluster), dim3(kAccThreads),
                          smem, stream, a);
}

// Node pass and finish with G 16-byte groups of the slice per thread
// (1 <= G <= kRejMaxG).
cudaError_t launch_reject(int G, const AcceptKArgs& a, int per, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_reject_g<1>(a, per, stream);
    case 2: return launch_reject_g<2>(a, per, stream);
    case 3: return launch_reject_g<3>(a, per, stream);
    case 4: return launch_reject_g<4>(a, per, stream);
    case 5: return launch_reject_g<5>(a, per, stream);
    case 6: return launch_reject_g<6>(a, per, stream);
    case 7: return launch_reject_g<7>(a, per, stream);
    case 8: return launch_reject_g<8>(a, per, stream);
    case 9: return launch_reject_g<9>(a, per, stream);
    default: return launch_reject_g<10>(a, per, stream);
  }
}
static_assert(kRejMaxG == 10, "one case per G");

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
  const int per = ((g.vocab + kAccCluster - 1) / kAccCluster + 3) & ~3;
  const int G = (per / 4 + kAccThreads - 1) / kAccThreads;
  if (g.mode == DS_ACCEPT_REJECT && g.n_nodes > 0 && a.vec && G <= kRejMaxG)
    return launch_reject(G, a, per, stream);   // node pass + finish (walk, bonus)
  cudaError_t e = cudaSuccess;
  if (g.n_nodes > 0) {
    if (g.mode != DS_ACCEPT_REJECT) {
      e = launch_dependent(accept_argmax, dim3(g.n_nodes * a.slices), dim3(kArgThreads), 0,
                           stream, a);
    } else {
      accept_reject_pass_stream<<<g.n_nodes * kAccCluster, kAccThreads, 0, stream>>>(a);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
  }
  return launch_dependent(accept_walk, dim3((g.batch + 3) / 4), dim3(128), 0, stream, a);
}

}  // namespace ds
