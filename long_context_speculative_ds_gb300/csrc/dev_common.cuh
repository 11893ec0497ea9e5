// Device-side helpers shared by the tree-verify kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "ds.h"
#include "internal.h"

#define DS_DEV __device__ __forceinline__

namespace ds {

constexpr int kTileKeys = 128;       // keys per attention tile
constexpr int kRowsPerGroup = DS_ROWS_PER_ITEM;   // query rows per work item
constexpr float kLog2e = 1.4426950408889634f;

DS_DEV void flag(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// ---------------------------------------------------------------------------
// Work plan of the split-KV verify pass.
//
// Sequence b contributes tiles_b = ceil((L_b + T_b) / 128) key tiles (context
// slots followed by its tree slots) for each of num_kv_heads heads and each
// row group of up to 256 query rows (rows = T_b * group).  All tile units of
// the batch are spread over about target_ctas work items: every (b, kv head,
// row group) is cut into splits_b = ceil(tiles_b / tps) contiguous tile
// ranges, tps = ceil(total_units / target_ctas).  Items are numbered
// sequence-major, then kv head, then row group, then split.  The plan is a
// pure function of (ctx_lens, tree_offsets, sizes), recomputed by every CTA
// that needs it, so no launch is spent on it and no host copy of the lengths
// is needed.
struct PlanArgs {
  const int32_t* ctx_lens;
  const int32_t* tree_offsets;
  int32_t batch, n_nodes, num_kv_heads, group, page_size, max_pages;
  int32_t chunk_size, max_chunks, target_ctas, rg_max;
  int32_t wave_ctas;    // > target_ctas: items a two-wave plan may use (0: one wave only)
  uint32_t* status;
};

struct SeqPlan {
  int32_t L, T, node0, tiles, rows, rg, splits, item_base;
};

struct Plan {
  int32_t tps;          // tiles per split
  int32_t total_items;
  SeqPlan seq;          // the sequence asked for (b_sel or item_sel)
  int32_t b;            // its index, -1 if none
};

// Validated per-sequence sizes; invalid sequences get T = 0 (no work).
DS_DEV SeqPlan seq_sizes(const PlanArgs& a, int b, bool report) {
  SeqPlan s;
  int32_t L = __ldg(a.ctx_lens + b);
  int32_t n0 = __ldg(a.tree_offsets + b);
  int32_t n1 = __ldg(a.tree_offsets + b + 1);
  int32_t T = n1 - n0;
  bool ok = true;
  if (L < 0 || (int64_t)L + (T > 0 ? T : 0) > (int64_t)a.max_pages * a.page_size ||
      (L + a.chunk_size - 1) / a.chunk_size > a.max_chunks) {
    ok = false;
    if (report) flag(a.status, DS_DEV_BAD_LENGTH);
  }
  if (T < 0 || T > DS_MAX_TREE_NODES || n0 < 0 || n1 > a.n_nodes) {
    ok = false;
    if (report) flag(a.status, DS_DEV_BAD_TREE);
  }
  s.L = ok ? L : 0;
  s.T = ok ? T : 0;
  s.node0 = ok ? n0 : 0;
  s.tiles = s.T > 0 ? (s.L + s.T + kTileKeys - 1) / kTileKeys : 0;
  s.rows = s.T * a.group;
  s.rg = (s.rows + kRowsPerGroup - 1) / kRowsPerGroup;
  s.splits = 0;
  s.item_base = 0;
  return s;
}

// Plan at tiles-per-split t (all 32 lanes of one warp): the prefix of items
// over the sequences, and the sequence asked for.
static __device__ __noinline__ Plan plan_at(const PlanArgs& a, int b_sel, int item_sel, int t) {
  const int lane = threadIdx.x & 31;
  Plan p;
  p.tps = t;
  p.b = -1;
  p.seq = SeqPlan{0, 0, 0, 0, 0, 0, 0, 0};
  int32_t base = 0;
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    int b = b0 + lane;
    SeqPlan s{0, 0, 0, 0, 0, 0, 0, 0};
    int32_t items = 0;
    if (b < a.batch) {
      s = seq_sizes(a, b, false);
      s.splits = (s.tiles + t - 1) / t;
      items = a.num_kv_heads * s.rg * s.splits;
    }
    int32_t incl = items;
    for (int o = 1; o < 32; o <<= 1) {
      int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    s.item_base = base + incl - items;
    bool hit = (b < a.batch) &&
               ((b_sel >= 0) ? (b == b_sel)
                             : (item_sel >= s.item_base && item_sel < s.item_base + items));
    unsigned m = __ballot_sync(0xffffffffu, hit);
    if (m) {
      int src = __ffs(m) - 1;
      p.b = __shfl_sync(0xffffffffu, b, src);
      p.seq.L = __shfl_sync(0xffffffffu, s.L, src);
      p.seq.T = __shfl_sync(0xffffffffu, s.T, src);
      p.seq.node0 = __shfl_sync(0xffffffffu, s.node0, src);
      p.seq.tiles = __shfl_sync(0xffffffffu, s.tiles, src);
      p.seq.rows = __shfl_sync(0xffffffffu, s.rows, src);
      p.seq.rg = __shfl_sync(0xffffffffu, s.rg, src);
      p.seq.splits = __shfl_sync(0xffffffffu, s.splits, src);
      p.seq.item_base = __shfl_sync(0xffffffffu, s.item_base, src);
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  p.total_items = base;
  return p;
}

// Splits round up per (sequence, kv head, row group), so ceil(total /
// target) tiles per split can need more items than there are CTAs, and the
// extra items would run as a second wave.  When the plan p does, this takes
// instead the smallest tiles-per-split whose items fit (when any does).
// When that split is more than 15 % above the one-wave ideal (p.tps on
// entry) and the grid has room for it (wave_ctas), the plan instead takes
// the smallest tiles-per-split whose items fit in wave_ctas: about two
// waves of half-size items, which the hardware hands to SMs as they free
// up, so the rounding of each group's split count costs less.
static __device__ __noinline__ Plan plan_refit(const PlanArgs& a, int b_sel, int item_sel,
                                               Plan p) {
  const int lane = threadIdx.x & 31;
  auto items_for = [&](int32_t t, int32_t& max_tiles) {
    int32_t it = 0;
    max_tiles = 0;
    for (int b0 = 0; b0 < a.batch; b0 += 32) {
      const int b = b0 + lane;
      int32_t v = 0, mt = 0;
      if (b < a.batch) {
        const SeqPlan s = seq_sizes(a, b, false);
        v = a.num_kv_heads * s.rg * ((s.tiles + t - 1) / t);
        mt = s.tiles;
      }
      for (int o = 16; o > 0; o >>= 1) {
        v += __shfl_xor_sync(0xffffffffu, v, o);
        mt = max(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      }
      it += v;
      max_tiles = max(max_tiles, mt);
    }
    return it;
  };
  int32_t max_tiles, unused;
  items_for(p.tps, max_tiles);
  if (max_tiles <= p.tps || items_for(max_tiles, unused) > a.target_ctas) return p;
  const int32_t ideal = p.tps;
  int32_t lo = p.tps, hi = max_tiles;   // items(lo) > target >= items(hi)
  while (hi - lo > 1) {
    const int32_t mid = lo + (hi - lo) / 2;
    if (items_for(mid, unused) <= a.target_ctas) hi = mid; else lo = mid;
  }
  if (a.wave_ctas > a.target_ctas && (int64_t)hi * 100 > (int64_t)ideal * 115) {
    // items(lo2) > wave_ctas >= items(hi2); hi2 = hi fits, since the
    // one-wave items do
    int32_t lo2 = max(1, ideal / 2) - 1, hi2 = hi;
    while (hi2 - lo2 > 1) {
      const int32_t mid = lo2 + (hi2 - lo2) / 2;
      if (items_for(mid, unused) <= a.wave_ctas) hi2 = mid; else lo2 = mid;
    }
    return plan_at(a, b_sel, item_sel, hi2);
  }
  return plan_at(a, b_sel, item_sel, hi);
}

// Must be called by all 32 lanes of one warp.  Finds the sequence with index
// b_sel (if b_sel >= 0) or the one owning work item item_sel.
DS_DEV Plan plan_find(const PlanArgs& a, int b_sel, int item_sel) {
  const int lane = threadIdx.x & 31;
  // pass 1: total tile units
  int64_t total = 0;
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    int b = b0 + lane;
    int64_t u = 0;
    if (b < a.batch) {
      SeqPlan s = seq_sizes(a, b, b_sel < 0 && item_sel == 0);
      u = (int64_t)s.tiles * a.num_kv_heads * s.rg;
    }
    for (int o = 16; o > 0; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
    total += u;
  }
  Plan p;
  int64_t tps = (total + a.target_ctas - 1) / (a.target_ctas > 0 ? a.target_ctas : 1);
  p.tps = (int32_t)(tps > 0 ? tps : 1);
  p.b = -1;
  p.seq = SeqPlan{0, 0, 0, 0, 0, 0, 0, 0};
  // pass 2: prefix of items
  int32_t base = 0;
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    int b = b0 + lane;
    SeqPlan s{0, 0, 0, 0, 0, 0, 0, 0};
    int32_t items = 0;
    if (b < a.batch) {
      s = seq_sizes(a, b, false);
      s.splits = (s.tiles + p.tps - 1) / p.tps;
      items = a.num_kv_heads * s.rg * s.splits;
    }
    int32_t incl = items;
    for (int o = 1; o < 32; o <<= 1) {
      int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    s.item_base = base + incl - items;
    bool hit = (b < a.batch) &&
               ((b_sel >= 0) ? (b == b_sel)
                             : (item_sel >= s.item_base && item_sel < s.item_base + items));
    unsigned m = __ballot_sync(0xffffffffu, hit);
    if (m) {
      int src = __ffs(m) - 1;
      p.b = __shfl_sync(0xffffffffu, b, src);
      p.seq.L = __shfl_sync(0xffffffffu, s.L, src);
      p.seq.T = __shfl_sync(0xffffffffu, s.T, src);
      p.seq.node0 = __shfl_sync(0xffffffffu, s.node0, src);
      p.seq.tiles = __shfl_sync(0xffffffffu, s.tiles, src);
      p.seq.rows = __shfl_sync(0xffffffffu, s.rows, src);
      p.seq.rg = __shfl_sync(0xffffffffu, s.rg, src);
      p.seq.splits = __shfl_sync(0xffffffffu, s.splits, src);
      p.seq.item_base = __shfl_sync(0xffffffffu, s.item_base, src);
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  p.total_items = base;
  if (p.total_items > a.target_ctas) p = plan_refit(a, b_sel, item_sel, p);
  return p;
}

// Ancestor mask of local node j (bit i set iff i is j or an ancestor of j),
// following parent links; invalid links (not an earlier node) stop the walk
// and are reported.
DS_DEV uint64_t ancestor_mask(const int32_t* parents_seq, int j, int T,
                              uint32_t* status) {
  uint64_t m = 0;
  int n = j;
  for (int guard = 0; guard <= DS_MAX_TREE_NODES && n >= 0; ++guard) {
    m |= 1ull << n;
    int p = __ldg(parents_seq + n);
    if (n == 0) {
      if (p != -1) flag(status, DS_DEV_BAD_TREE);
      break;
    }
    if (p < 0 || p >= n) {
      flag(status, DS_DEV_BAD_TREE);
      break;
    }
    n = p;
  }
  (void)T;
  return m;
}

DS_DEV float warp_max(float v) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
DS_DEV float warp_sum(float v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
DS_DEV double warp_sum_d(double v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace ds
