// Host-side internals shared by the ABI layer and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ds.h"

namespace ds {

#ifndef DS_ROWS_PER_ITEM
#define DS_ROWS_PER_ITEM 256
#endif
// query rows per split-pass work item (128 or 256)
constexpr int kRowsPerItem = DS_ROWS_PER_ITEM;

constexpr size_t kAlign = 256;
constexpr size_t kStatusBytes = 256;   // status word region at workspace start

inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

// Workspace layout of ds_verify_attn (byte offsets from the workspace start).
struct VerifyLayout {
  int32_t group;        // num_q_heads / num_kv_heads
  int32_t rg_max;       // row groups per (sequence, kv head) at 64 nodes
  int32_t target_ctas;  // CTAs the plan aims at
  int32_t wave_ctas;    // items a two-wave plan may use (batches of more than one sequence; 0: none)
  int32_t max_items;    // upper bound on work items
  size_t counters;      // [batch][kv][rg_max] u32           splits finished (0 between calls)
  size_t gdesc;         // [batch][kv][rg_max] int4          first item and splits of the
                        //                                   row group (by its last split)
  size_t o_part;        // [max_items][256][head_dim] split outputs (normalised), bf16
                        // when the output is bf16, else f32 (sized for f32)
  size_t lse_part;      // [max_items][256] f32              split log2-sum-exp
  size_t clse;          // [batch][kv][rg_max][max_chunks][256] f32 chunk log2 mass
  size_t row_lse;       // [batch][kv][rg_max][256] f32      final row log2-sum-exp
  size_t total;
};

struct AcceptLayout {
  size_t node_stats;    // [n_nodes] NodeStats
  size_t total;
};

// Slices of the vocabulary into which the greedy argmax pass cuts a node's
// target row (one CTA each).
constexpr int kArgmaxSlices = 8;

// Slices of the greedy argmax pass for a vocabulary: about 4096 logits or more
// per CTA, at most kArgmaxSlices.
inline int accept_argmax_slices(int vocab) {
  const int s = (vocab + 4095) / 4096;
  return s < 1 ? 1 : (s > kArgmaxSlices ? kArgmaxSlices : s);
}

// Per-node statistics written by the acceptance node passes.  The rejection
// fields are the fp32 scalars the node pass itself used, so that the walk
// evaluates p(x), q(x) and the residual chain at a token with exactly the
// node pass's float operations.
struct NodeStats {
  float m_t, inv_s_t;   // target: max logit, 1 / sum exp(l - max)   (rejection)
  float m_d, inv_s_d;   // draft:  the same                          (rejection)
  // bonus distribution if the walk stops here after rejecting every child:
  // proportional to max(0, p - s_bonus q)          (rejection, inner node)
  float s_bonus;
  int32_t bonus_stop;   // bonus token if the walk stops here  (streaming pass)
  // 1 when this node, as a child, passes its test u * q(x) < r(x) at its
  // parent, r the residual after its elder siblings were rejected (rejection)
  int32_t pass;
  int32_t pad_;
  uint64_t amax[kArgmaxSlices];   // greedy: per slice, the largest key
                                  // (order-preserving bits of the logit << 32
                                  // | ~index), so the maximum key is the
                                  // largest logit at its lowest index
};
static_assert(sizeof(NodeStats) == 96, "the record size ds.h states for ds_accept_static");


VerifyLayout verify_layout(const ds_verify_args& a, int num_sms);
AcceptLayout accept_layout(const ds_accept_args& a);

// Launchers (return cudaSuccess or the launch error).
cudaError_t launch_verify(const ds_verify_args& a, const VerifyLayout& L,
                          cudaStream_t stream);
cudaError_t launch_topk_gather(const ds_gather_args& a, cudaStream_t stream);
cudaError_t launch_accept(const ds_accept_args& a, const AcceptLayout& L,
                          cudaStream_t stream);

cudaError_t launch_kv_commit(const ds_commit_args& a, cudaStream_t stream);
cudaError_t launch_compact_append(const ds_append_args& a, cudaStream_t stream);

// Sets the message ds_last_error returns on this thread; returns st.
ds_status set_last_error(ds_status st, const char* msg);

}  // namespace ds
