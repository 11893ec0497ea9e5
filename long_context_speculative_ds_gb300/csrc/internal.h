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
  int32_t max_items;    // upper bound on work items
  size_t o_part;        // [max_items][256][head_dim] f32   split outputs (normalised)
  size_t lse_part;      // [max_items][256] f32              split log2-sum-exp
  size_t clse;          // [batch][kv][rg_max][max_chunks][256] f32 chunk log2 mass
  size_t row_lse;       // [batch][kv][rg_max][256] f32      final row log2-sum-exp
  size_t total;
};

struct AcceptLayout {
  size_t node_stats;    // [n_nodes] NodeStats
  size_t total;
};

// Per-node statistics written by the acceptance node pass.
struct NodeStats {
  double m_t, s_t;      // target: max logit, sum exp(l - m)
  double m_d, s_d;      // draft:  max logit, sum exp(l - m)
  double z_after;       // residual normaliser after rejecting this node (as a child)
  int32_t argmax_t;     // lowest index of the target maximum
  int32_t bonus_stop;   // bonus token if the walk stops at this node (rejection)
};

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
