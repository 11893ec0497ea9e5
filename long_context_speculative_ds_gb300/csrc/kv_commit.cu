// Post-accept KV commit (adaptive-specdec README, "Layout": one cache buffer
// per layer, a per-sequence lengths vector, writes scattered to each row's
// own offset, rollback by length).
//
// The accepted nodes c_1 < ... < c_n of sequence b move from tree slots
// L + c_i to L + i, K and V, in every layer and kv head; the new length is
// L + 1 + n (the root, node 0, already sits at slot L).
//
// One CTA per (tensor K or V, kv head, layer, sequence): it reads all n
// source rows of its head into shared memory, then writes them to their
// destinations.  Reading everything first matters: a destination slot L + i
// can be the source slot of an earlier path entry (c_k = i for some k < i).
// CTAs never touch each other's rows (different head, tensor or layer).
#include <cuda_runtime.h>
#include <stdint.h>

#include "dev_common.cuh"
#include "internal.h"

namespace ds {

struct CommitKArgs {
  const void* k[DS_MAX_COMMIT_LAYERS];
  const void* v[DS_MAX_COMMIT_LAYERS];
  const int32_t* page_table;
  const int32_t* ctx_lens;
  const int32_t* offsets;
  const int32_t* path;
  const int32_t* n_acc;
  int32_t batch, num_kv_heads, head_dim, page_size, num_pages, max_pages;
  int64_t page_stride, tok_stride, head_stride;   // elements
  int32_t* new_lens;
  uint32_t* status;
};

constexpr int kCommitThreads = 256;

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(const CommitKArgs a) {
  // rows of up to 63 accepted nodes x head_dim bf16 (<= 16 KB)
  __shared__ uint4 rows[(DS_MAX_TREE_NODES - 1) * 128 * 2 / 16];
  __shared__ int s_nodes[DS_MAX_TREE_NODES];
  __shared__ int s_n, s_ok;
  const int tensor = blockIdx.x & 1, h = blockIdx.x >> 1;
  const int layer = blockIdx.y, b = blockIdx.z;
  const int L = __ldg(a.ctx_lens + b);
  const int n0 = __ldg(a.offsets + b), n1 = __ldg(a.offsets + b + 1);
  const int T = n1 - n0;
  const bool first = blockIdx.x == 0 && layer == 0;   // reports and writes the length

  // sequence checks; warp 0 loads the path lane-parallel and checks that
  // it is strictly increasing inside (0, T)
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int n = __ldg(a.n_acc + b);
    int ok = 1;          // 1: commit, 0: nothing to move
    int len = L;
    if (L < 0) {
      ok = 0;
      if (first && lane == 0) flag(a.status, DS_DEV_BAD_LENGTH);
    } else if (T < 0 || T > DS_MAX_TREE_NODES) {
      ok = 0;
      if (first && lane == 0) flag(a.status, DS_DEV_BAD_TREE);
    } else if (T == 0) {
      ok = 0;
    } else if ((int64_t)L + T > (int64_t)a.max_pages * a.page_size) {
      ok = 0;
      if (first && lane == 0) flag(a.status, DS_DEV_BAD_LENGTH);
    } else {
      bool good = n >= 0 && n <= T - 1;
      if (good) {
        const int32_t* pp = a.path + (int64_t)b * DS_MAX_TREE_NODES;
        const int c0 = lane < n ? __ldg(pp + lane) : 0;
        const int c1 = lane + 32 < n ? __ldg(pp + lane + 32) : 0;
        // every lane takes part in every shuffle (none sits in a branch)
        const int up0 = __shfl_up_sync(0xffffffffu, c0, 1);
        const int up1 = __shfl_up_sync(0xffffffffu, c1, 1);
        const int last0 = __shfl_sync(0xffffffffu, c0, 31);
        const int prev0 = lane == 0 ? 0 : up0;
        const int prev1 = lane == 0 ? last0 : up1;
        const bool bad0 = lane < n && !(c0 > prev0 && c0 < T);
        const bool bad1 = lane + 32 < n && !(c1 > prev1 && c1 < T);
        good = !__any_sync(0xffffffffu, bad0 || bad1);
        if (lane < n) s_nodes[lane] = c0;
        if (lane + 32 < n) s_nodes[lane + 32] = c1;
      }
      if (!good) {
        if (first && lane == 0) flag(a.status, DS_DEV_BAD_TREE);
        n = 0;         // the root is committed, the path is not
      }
      len = L + 1 + n;
    }
    if (lane == 0) {
      s_ok = ok;
      s_n = ok ? n : 0;
      if (first) a.new_lens[b] = len;
    }
  }
  __syncthreads();
  const int n = s_n;
  if (!s_ok || n == 0) return;

  const int32_t* pt = a.page_table + (int64_t)b * a.max_pages;
  const uint4* src = reinterpret_cast<const uint4*>(tensor ? a.v[layer] : a.k[layer]);
  uint4* dst = reinterpret_cast<uint4*>(const_cast<void*>(tensor ? a.v[layer] : a.k[layer]));
  const int vpr = a.head_dim / 8;                    // 16-byte vectors per row
  // element offset of (slot, head h) or -1 for an invalid page
  auto row_off = [&](int slot) -> int64_t {
    const int pg = __ldg(pt + slot / a.page_size);
    if (pg < 0 || pg >= a.num_pages) return -1;
    return (int64_t)pg * a.page_stride + (int64_t)(slot % a.page_size) * a.tok_stride +
           (int64_t)h * a.head_stride;
  };
  const int total = n * vpr;
  for (int e = threadIdx.x; e < total; e += kCommitThreads) {
    const int i = e / vpr, c = e % vpr;
    const int64_t off = row_off(L + s_nodes[i]);
    rows[e] = off >= 0 ? src[off / 8 + c] : make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < total; e += kCommitThreads) {
    const int i = e / vpr, c = e % vpr;
    const int64_t so = row_off(L + s_nodes[i]);
    const int64_t off = row_off(L + 1 + i);
    if (so < 0 || off < 0) {
      if (c == 0) flag(a.status, DS_DEV_BAD_PAGE);
      continue;
    }
    dst[off / 8 + c] = rows[e];
  }
}

cudaError_t launch_kv_commit(const ds_commit_args& g, cudaStream_t stream) {
  CommitKArgs a;
  for (int l = 0; l < DS_MAX_COMMIT_LAYERS; ++l) {
    a.k[l] = l < g.num_layers ? g.k_caches[l] : nullptr;
    a.v[l] = l < g.num_layers ? g.v_caches[l] : nullptr;
  }
  a.page_table = g.page_table;
  a.ctx_lens = g.ctx_lens;
  a.offsets = g.tree_offsets;
  a.path = g.path;
  a.n_acc = g.n_accepted;
  a.batch = g.batch;
  a.num_kv_heads = g.num_kv_heads;
  a.head_dim = g.head_dim;
  a.page_size = g.page_size;
  a.num_pages = g.num_pages;
  a.max_pages = g.max_pages;
  const int64_t P = g.page_size, H = g.num_kv_heads, D = g.head_dim;
  if (g.kv_layout == DS_KV_NHD) {
    a.page_stride = P * H * D; a.tok_stride = H * D; a.head_stride = D;
  } else {
    a.page_stride = H * P * D; a.tok_stride = D; a.head_stride = P * D;
  }
  a.new_lens = g.new_ctx_lens;
  a.status = static_cast<uint32_t*>(g.workspace);
  const dim3 grid(2 * g.num_kv_heads, g.num_layers, g.batch);
  kv_commit_kernel<<<grid, kCommitThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ds
