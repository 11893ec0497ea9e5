// Tree acceptance: greedy accept-if-equal or exact tree rejection sampling
// (vllm.cpp docs "Speculative decoding", MTP; adaptive-specdec README,
// "Correctness first" and "The controller").
//
// node pass (one thread-block cluster of 8 CTAs per tree node, each CTA one
//   eighth of the vocabulary, partial results combined through distributed
//   shared memory):
//     target max and its lowest index (greedy stops here);
//     sum exp(l - max) for target and draft;
//     for the k-th child of the node, the residual normaliser
//       Z_k = sum_y max(0, r_{k-1}(y) - q(y)),  r_0 = p,
//       r_k = max(0, r_{k-1} - q) / Z_k  (r_k = r_{k-1} when Z_k = 0),
//     which does not depend on the children's tokens, so every node's
//     residual chain is computed in parallel before the walk;
//     the bonus token the walk would draw if it stopped here: the smallest x
//     with sum_{y<=x} r_m(y) > u * sum_y r_m(y), m = number of children.
//   Per-element values are fp32; sums use compensated fp32 per thread and
//   float64 across threads.
// walk (one warp per sequence): follows the tree from the root.  Greedy
//   compares draft tokens with the stored argmax; rejection evaluates p(x),
//   q(x) and the residual chain at the proposed token in float64 from the
//   stored normalisers and tests u * q(x) < r(x).
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "dev_common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace ds {

constexpr int kAccCluster = 8;
constexpr int kAccThreads = 512;
constexpr int kAccWarps = kAccThreads / 32;

struct AcceptKArgs {
  int32_t mode;
  const float* tl;
  const float* dl;
  const int32_t* tokens;
  const int32_t* parents;
  const int32_t* offsets;
  const float* uniforms;
  int32_t batch, n_nodes, vocab;
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
accept_node_pass(AcceptKArgs a) {
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
  const bool reject = a.mode == DS_ACCEPT_REJECT;
  const float* drow = reject ? a.dl + (int64_t)node * V : nullptr;
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
  if (!reject) {
    if (rank == 0 && threadIdx.x == 0) a.stats[node].argmax_t = I;
    return;
  }

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
    if (rank == 0 && threadIdx.x == 0) a.stats[n0 + s_children[k]].z_after = Z;
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
    a.stats[node].argmax_t = I;
    a.stats[node].m_t = M;
    a.stats[node].s_t = St;
    a.stats[node].m_d = Md;
    a.stats[node].s_d = Sd;
  }
  cl.sync();
}

// One warp per sequence.
__global__ void __launch_bounds__(128) accept_walk(AcceptKArgs a) {
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
      const int y = a.stats[n0 + i].argmax_t;
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
          const double p = exp((double)__ldg(a.tl + (int64_t)(n0 + i) * V + x) - st.m_t) / st.s_t;
          const double q = exp((double)__ldg(a.dl + (int64_t)(n0 + i) * V + x) - st.m_d) / st.s_d;
          double r = p;
          uint64_t rj = rejected;
          while (rj) {
            const int cj = __ffsll((long long)rj) - 1;
            rj &= rj - 1;
            const double z = a.stats[n0 + cj].z_after;
            if (z > 0.0) r = fmax(0.0, r - q) / z;
          }
          const double u = (double)__ldg(a.uniforms + 2 * (int64_t)(n0 + c));
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
  if (lane == 0) {
    a.out_n[b] = n;
    a.out_bonus[b] = reject ? a.stats[n0 + i].bonus_stop : a.stats[n0 + i].argmax_t;
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
  unsigned char* ws = static_cast<unsigned char*>(g.workspace);
  a.stats = reinterpret_cast<NodeStats*>(ws + L.node_stats);
  a.out_path = g.out_path;
  a.out_n = g.out_n_accepted;
  a.out_bonus = g.out_bonus;
  a.status = reinterpret_cast<uint32_t*>(ws);
  if (g.n_nodes > 0) {
    accept_node_pass<<<g.n_nodes * kAccCluster, kAccThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  accept_walk<<<(g.batch + 3) / 4, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ds
