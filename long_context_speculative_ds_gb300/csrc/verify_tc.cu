// Split pass of the tree-verify attention on the 5th-generation tensor cores
// (tcgen05) of sm_103a.
//
// One CTA per work item (sequence, kv head, row group of up to 256 query
// rows, contiguous range of 128-key tiles), 12 warps:
//   warp 0      loader: Q once, then K and V tiles into shared-memory rings.
//               Pages wholly inside the sequence arrive by TMA, one box per
//               page (all columns of one kv head: a 5-D tensor map lands it
//               as [8-row group][64-column half][8 rows x 128 B], whole
//               128-byte-swizzle atoms); the one page that holds the
//               sequence end is copied with plain loads so that slots past
//               the end read as zero, and pages wholly past the end get an
//               out-of-range coordinate (TMA fills zeros).
//   warp 1      tensor-memory allocator; in the split that holds the tree's
//               keys it then forms the tree's ancestor masks, beside the
//               loader, for the softmax warps' tree units.
//   warps 2, 3  MMA issuers of softmax groups 0 and 1 (one thread each).
//   warps 4-7   softmax group 0, warps 8-11 softmax group 1 (each a whole
//               warpgroup): one query row per thread, tensor-memory lane
//               32 * (warp % 4) + lane.
//
// Each softmax group owns a stream of 128-key tiles: with more than 128
// rows group g takes rows 128g..128g+127 of every tile ("row mode"); with at
// most 128 rows both groups use the same rows and take alternate tiles, and
// their partial results are merged at the end ("key mode").  Tensor memory,
// 256 columns per group: two 64-column half slots and O (128 columns).
// Half slot h holds S = Q K^T of keys 64h..64h+63 of the group's tile (one
// M128 N64 chain), which the group turns into bf16 P in place and signals;
// the group's issuer then issues O += P V for that half and, into the same
// slot (the pipe runs in order), S of the same half of the group's next
// tile.  So each half's S is ready long before the group gets to it, and
// the two groups keep the tensor pipe busy while either computes
// exponentials.  A thread that has issued tcgen05.mma pays for its own
// next shared-memory access (a barrier test included) with the time its
// queued MMAs take to drain; with one issuer per group, each issuer waits
// only for its own group's P, by which time its MMAs have completed.
//
// Softmax works in log2 units with lazy rescaling: the running maximum only
// moves (and O is rescaled, after the previous P V has completed) when a
// row's new maximum exceeds it by more than 8, so P stays below 2^8.  For
// every context chunk each row also writes log2 of the chunk's attention
// mass relative to the row's maximum (plus that maximum); the finalize kernel
// turns these into chunk salience.  Tree keys count toward the softmax
// denominator only.
//
// Every wait is bounded; on a timeout the CTA raises DS_DEV_TIMEOUT, drains
// what it issued, frees its tensor memory and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "dev_common.cuh"
#include "internal.h"
#include "pdl.cuh"
#include "tc_ptx.cuh"
#include "verify_common.cuh"

namespace ds {
namespace tc {

constexpr int kThreads = 384;
// Q tiles: [column half][128 rows x 128 bytes (64 bf16)]
constexpr uint32_t kHalfBytes = 128 * 128;
constexpr int kTmemCols = 512;

enum Bar {
  kQFull = 0,
  kKFull = 1,      // [group][slot] in key mode, [0][slot] in row mode
  kKEmpty = 7,     // 3 slots
  kVFull = 10,     // [group][slot] in key mode, [0][slot] in row mode
  kVEmpty = 16,    // 3 slots
  kSFull = 19,     // [group][half]: S of the group's next 64-key half is
                   // ready in that half's tensor-memory slot
  kPFull = 23,     // [group][half]: P of one 64-key half is ready; one
                   // barrier per half, so that a group can never complete
                   // two phases of one barrier before the MMA thread has
                   // seen the first
  kORdy = 27,      // [group]: one completion per issued P V
  kOFinal = 29,    // [group]: all of the group's MMAs have completed
  kAnc = 31,       // the tree's ancestor masks are in ctrl->anc (warp 1)
  kNumBars = 32
};

struct Ctrl {
  uint64_t bar[kNumBars];
  uint32_t tmem_base;
  int abort;
  Plan plan;
  int32_t parents[DS_MAX_TREE_NODES];
  uint64_t anc[DS_MAX_TREE_NODES];
  uint32_t where[5];   // last wait site of loader, issuer 0, softmax 0, softmax 1, issuer 1
  int last;            // this CTA is the last split of its row group to finish
};

template <int D>
struct Cfg {
  static constexpr int TB = 128 * D * 2;   // bytes of one 128-row tile
  static constexpr int NH = D / 64;        // 128-byte column halves
  // K and V tiles: [row group of 8 keys][column half][8 rows x 128 bytes],
  // so that one page of P keys (P / 8 row groups, all columns) is one
  // contiguous P * D * 2-byte block that a single TMA box fills; each
  // 1 KB block of 8 rows x 128 bytes is one 128-byte-swizzle atom
  static constexpr uint32_t RG = NH * 1024;   // bytes of one row group
  // Q (2 tiles) + K ring (2 slots) + V ring (3 slots) + control block
  static constexpr size_t smem = 7 * TB + sizeof(Ctrl) + 1024;
  static_assert(smem <= 232448, "dynamic shared memory above the 227 KB a block can have");
  // the epilogue stages four warps' 32 x 32-float tiles inside one Q tile
  static_assert(4 * 32 * 32 * 4 <= TB, "output staging must fit in a Q tile");
};

// One 64-key unit of one softmax thread (one query row): loads the row's 64
// scores from tensor memory, applies the tree/tail mask (TAIL only), updates
// the running maximum lazily, writes the exponentials as bf16 P over the
// first 32 columns of the buffer, and emits the log2 attention mass of every
// context chunk that ends in this unit.  `cs` carries the context mass of a
// chunk that started in the previous unit of the same tile.  Returns the
// factor by which O must be scaled (alpha) and whether any row of the warp
// needs it.
template <bool TAIL>
DS_DEV void softmax_unit(const uint32_t tS, const uint32_t tP, const uint32_t vw0,
                         const uint32_t vw1,
                         const uint32_t cw0, const uint32_t cw1, const float c2, const bool first,
                         float& m2, float& l, float& cs, float& alpha, bool& rescale,
                         const int tile_slot0, const int kbase, const int cshift, const int n_ch,
                         const bool row_ok, float* __restrict__ clse_row) {
  using namespace ptx;
  float s[64];
  {
    uint32_t r0[32], r1[32];
    tmem_ld32(tS, r0);
    tmem_ld32(tS + 32, r1);
    tmem_ld_wait(r0);
    tmem_ld_wait(r1);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      s[i] = __uint_as_float(r0[i]);
      s[32 + i] = __uint_as_float(r1[i]);
    }
  }
  if constexpr (TAIL) {
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      if (!((vw0 >> c) & 1u)) s[c] = -CUDART_INF_F;
      if (!((vw1 >> c) & 1u)) s[32 + c] = -CUDART_INF_F;
    }
  }
  // row maximum: three-input max, four independent chains of 16
  float mx4[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float m = fmax3(s[16 * k], s[16 * k + 1], s[16 * k + 2]);
#pragma unroll
    for (int i = 3; i < 15; i += 2) m = fmax3(m, s[16 * k + i], s[16 * k + i + 1]);
    mx4[k] = fmaxf(m, s[16 * k + 15]);
  }
  const float mx2 = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3])) * c2;
  alpha = 1.f;
  rescale = false;
  if (first) {
    m2 = mx2;
  } else {
    const bool need = mx2 > m2 + 8.f;
    rescale = __any_sync(0xffffffffu, need);
    if (need) {
      alpha = ex2(m2 - mx2);
      m2 = mx2;
    }
  }
  const float mb = (m2 == -CUDART_INF_F) ? 0.f : m2;
  // exponentials (masked columns: ex2(-inf) = 0) and per-16-column sums of
  // the context columns; tree columns of a tail unit go to tsum
  float cg[4];
  float tsum = 0.f;
  if constexpr (TAIL) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const int c = 16 * k + i;
        const float e0 = ex2(fmaf(s[c], c2, -mb));
        const float e1 = ex2(fmaf(s[c + 1], c2, -mb));
        s[c] = e0;
        s[c + 1] = e1;
        const uint32_t w = c < 32 ? cw0 : cw1;
        const bool k0 = (w >> (c & 31)) & 1u;
        const bool k1 = (w >> ((c + 1) & 31)) & 1u;
        a0 += k0 ? e0 : 0.f;
        a1 += k1 ? e1 : 0.f;
        tsum += (k0 ? 0.f : e0) + (k1 ? 0.f : e1);
      }
      cg[k] = a0 + a1;
    }
  } else {
    // pairs of columns in f32x2 arithmetic: (s c2 - mb) and the running sums
    const uint64_t c2x2 = f2pack(c2, c2), nmb2 = f2pack(-mb, -mb);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint64_t acc = f2pack(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const int c = 16 * k + i;
        float x0, x1;
        f2unpack(ffma2(f2pack(s[c], s[c + 1]), c2x2, nmb2), x0, x1);
        s[c] = ex2(x0);
        s[c + 1] = ex2(x1);
        acc = fadd2(acc, f2pack(s[c], s[c + 1]));
      }
      float lo, hi;
      f2unpack(acc, lo, hi);
      cg[k] = lo + hi;
    }
  }
  l = l * alpha + (tsum + ((cg[0] + cg[1]) + (cg[2] + cg[3])));
  // chunk log2-mass at chunk boundaries (C/16 sixteen-column groups a chunk)
  {
    const int per_mask = (1 << (cshift - 4)) - 1;
    cs *= alpha;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      cs += cg[k];
      const int kg = kbase + k;          // 16-column group index in the tile
      if (((kg + 1) & per_mask) == 0) {
        const int cidx = (tile_slot0 + kg * 16) >> cshift;
        if (row_ok && cidx < n_ch)
          clse_row[(int64_t)cidx * kRowsPerGroup] = cs > 0.f ? mb + __log2f(cs) : -CUDART_INF_F;
        cs = 0.f;
      }
    }
  }
  // P as bf16 pairs (keys 2i, 2i+1 -> column i of tP)
  uint32_t pk[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(s[2 * i], s[2 * i + 1]);
  tmem_st32(tP, pk);
}

// Output of one softmax thread after its last tile: O / l (merged with the
// other group's partial result in key mode) and the row's log2-sum-exp.
// The rows are written through a per-warp staging tile in shared memory
// (`stage`, 32 rows x 32 floats = 4 KB, idle by then; 16-byte chunk c of row
// r stored at chunk c ^ (r % 8), so that eight consecutive lanes touch all
// 32 banks both when a thread writes its row and when a lane reads a row
// segment): each thread writes its row's 32-column slice, then each warp
// store writes four rows' 128-byte segments, so the global writes are whole
// segments instead of 32 rows' scattered 16 bytes.
constexpr int kStageStride = 32;   // floats per staged row

template <int D>
__device__ __noinline__ void write_row_output(const bool row_mode, const int g, const bool ok,
                                              const int nt1, const uint32_t tO, const int lrow,
                                              const int rows_left, const float m2,
                                              const float l, float* __restrict__ merge_buf,
                                              float* m1buf, float* l1buf,
                                              float* __restrict__ stage,
                                              const bool part_bf16,
                                              void* __restrict__ op_warp,
                                              float* __restrict__ lse_out) {
  using namespace ptx;
  const int lane = threadIdx.x & 31;
  const bool row_ok = (lrow & 31) < rows_left;
  if (!row_mode && g == 1) {
    if (ok && nt1 > 0) {
#pragma unroll 1
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t r[32];
        tmem_ld32(tO + c4 * 32, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) merge_buf[(c4 * 32 + i) * 128 + lrow] = __uint_as_float(r[i]);
      }
    }
    m1buf[lrow] = m2;
    l1buf[lrow] = l;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    return;
  }
  float sc0 = 1.f, sc1 = 0.f, lt = l, mt = m2;
  if (!row_mode) {
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (nt1 > 0) {
      const float m1 = m1buf[lrow], l1 = l1buf[lrow];
      mt = fmaxf(m2, m1);
      const float mb2 = (mt == -CUDART_INF_F) ? 0.f : mt;
      sc0 = l > 0.f ? ex2(m2 - mb2) : 0.f;
      sc1 = l1 > 0.f ? ex2(m1 - mb2) : 0.f;
      lt = l * sc0 + l1 * sc1;
    }
  }
  const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll 1
  for (int c4 = 0; c4 < D / 32; ++c4) {
    uint32_t r[32];
    if (ok) {
      tmem_ld32(tO + c4 * 32, r);
      tmem_ld_wait(r);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = 0u;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float o = __uint_as_float(r[i]) * sc0;
      if (sc1 != 0.f) o += merge_buf[(c4 * 32 + i) * 128 + lrow] * sc1;
      r[i] = __float_as_uint(o * inv);
    }
    if (part_bf16) {
      // bf16 pairs: a row's 32 columns are 64 bytes, four 16-byte chunks;
      // chunk c of row q sits in the row's slot c ^ ((q / 2) % 4), so that
      // eight lanes of one access (eight rows, or two rows' four chunks)
      // touch distinct 16-byte bank groups
      uint32_t* st = reinterpret_cast<uint32_t*>(stage) + lane * 16;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[e] = pack_bf16x2(__uint_as_float(r[8 * c + 2 * e]),
                             __uint_as_float(r[8 * c + 2 * e + 1]));
        *reinterpret_cast<uint4*>(st + 4 * (c ^ ((lane >> 1) & 3))) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
      __syncwarp();
      // rows 8k + lane / 4, 16-byte chunk lane % 4 of the slice
      __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(op_warp);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int rr = 8 * k + (lane >> 2), cc = lane & 3;
        if (rr < rows_left) {
          const uint4 v = *reinterpret_cast<const uint4*>(
              reinterpret_cast<const uint32_t*>(stage) + rr * 16 + 4 * (cc ^ ((rr >> 1) & 3)));
          *reinterpret_cast<uint4*>(ob + (int64_t)rr * D + c4 * 32 + cc * 8) = v;
        }
      }
      __syncwarp();
      continue;
    }
    // f32: this thread's row, 32 columns, into the staging tile
#pragma unroll
    for (int i = 0; i < 32; i += 4)
      *reinterpret_cast<float4*>(stage + lane * kStageStride + 4 * ((i >> 2) ^ (lane & 7))) =
          make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                      __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
    __syncwarp();
    // rows 4k + lane / 8, columns 4 (lane % 8) .. + 3 of the slice
    float* of = reinterpret_cast<float*>(op_warp);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int rr = 4 * k + (lane >> 3), cc = 4 * (lane & 7);
      if (rr < rows_left) {
        const float4 v = *reinterpret_cast<const float4*>(
            stage + rr * kStageStride + 4 * ((lane & 7) ^ (rr & 7)));
        *reinterpret_cast<float4*>(of + (int64_t)rr * D + c4 * 32 + cc) = v;
      }
    }
    __syncwarp();
  }
  if (row_ok) *lse_out = lt > 0.f ? mt + __log2f(lt) : -CUDART_INF_F;
}

// Final log2-sum-exp of one row from its ns splits' (lp[s * 256]): 32 loads
// at a time, merged as a running (max, sum of 2^(x - max)).
DS_DEV float row_lse_from_splits(const float* lp, int ns) {
  constexpr int kB = 32;
  float mx = -CUDART_INF_F, sum = 0.f;
  for (int s0 = 0; s0 < ns; s0 += kB) {
    float v[kB];
#pragma unroll
    for (int k = 0; k < kB; ++k)
      v[k] = s0 + k < ns ? __ldcg(lp + (int64_t)(s0 + k) * kRowsPerGroup) : -CUDART_INF_F;
    float bm = v[0];
#pragma unroll
    for (int k = 1; k < kB; ++k) bm = fmaxf(bm, v[k]);
    const float nm = fmaxf(mx, bm);
    if (nm == -CUDART_INF_F) continue;
    float add = 0.f;
#pragma unroll
    for (int k = 0; k < kB; ++k) add += exp2f(v[k] - nm);
    sum = (mx == -CUDART_INF_F ? 0.f : sum * exp2f(mx - nm)) + add;
    mx = nm;
  }
  return sum > 0.f ? mx + log2f(sum) : -CUDART_INF_F;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    verify_split_tc(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const VerifyKArgs a,
                    const int hnd) {
  using namespace ptx;
  constexpr int TB = Cfg<D>::TB;
  constexpr int NH = Cfg<D>::NH;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t sQ = sbase;             // Q tiles 0, 1
  const uint32_t sK = sbase + 2 * TB;    // K slots 0, 1 (slot 2 = Q tile 1 in key mode)
  const uint32_t sV = sbase + 4 * TB;    // V slots 0, 1, 2
  // key-mode merge scratch, used once the V ring is idle: O of group 1
  // [D][128] f32 and its row maxima and sums
  float* merge_buf = reinterpret_cast<float*>(smem + 4 * TB);
  float* m1buf = reinterpret_cast<float*>(smem + 6 * TB);
  float* l1buf = m1buf + 128;
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + 7 * TB);
  volatile int* abort_flag = &ctrl->abort;
  uint32_t* diag = a.plan.status + 1;   // where a bounded wait gave up

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) { return smem_addr(&ctrl->bar[i]); };

  // ---------------------------------------------------------------- set-up
  // Barriers and tensor memory touch no global memory, so they are set up
  // before waiting for the preceding kernel of the stream; everything that
  // reads the call's inputs comes after the wait, except, for a call that
  // accumulates scores (a later layer of the same step), the work plan: its
  // inputs (lengths, tree offsets) are the step's, which the kernel right
  // before such a call does not write, so the search overlaps its tail.
  if (warp == 1 && lane == 0) {
    mbar_init(bar(kQFull), 1);
    for (int s = 0; s < 6; ++s) {
      mbar_init(bar(kKFull + s), 1);
      mbar_init(bar(kVFull + s), 1);
    }
    for (int s = 0; s < 3; ++s) {
      mbar_init(bar(kKEmpty + s), 2);   // one commit per group (two in key mode)
      mbar_init(bar(kVEmpty + s), 2);
    }
    for (int s = 0; s < 2; ++s) mbar_init(bar(kORdy + s), 1);
    for (int s = 0; s < 4; ++s) mbar_init(bar(kSFull + s), 1);
    for (int s = 0; s < 4; ++s) mbar_init(bar(kPFull + s), 128);
    for (int s = 0; s < 2; ++s) mbar_init(bar(kOFinal + s), 1);
    mbar_init(bar(kAnc), 32);
    ctrl->abort = 0;
    for (int i = 0; i < 5; ++i) ctrl->where[i] = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&ctrl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  const bool early_plan = a.accumulate != 0;
  if (early_plan && warp == 0) {
    Plan p = plan_find(a.plan, -1, blockIdx.x);
    if (lane == 0) ctrl->plan = p;
  }
  grid_dep_wait();
  grid_dep_launch_dependents();
  if (!early_plan && warp == 0) {
    Plan p = plan_find(a.plan, -1, blockIdx.x);
    if (lane == 0) ctrl->plan = p;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  const Plan p = ctrl->plan;
  const bool active = (int)blockIdx.x < p.total_items && p.b >= 0;

  // work item
  const SeqPlan& sq = p.seq;
  const int G = a.plan.group;
  int kvh = 0, rgi = 0, t0 = 0, t1 = 0, rows_here = 0;
  if (active) {
    const int local = blockIdx.x - sq.item_base;
    const int per_h = sq.rg * sq.splits;
    kvh = local / per_h;
    rgi = (local % per_h) / sq.splits;
    // The sequence's tiles in sq.splits near-equal ranges, the larger ones
    // first (the last range holds the tree's tile): the split count comes
    // from the plan's tiles per split, without full splits and a short
    // remainder.
    const int split = local % sq.splits;
    const int base = sq.tiles / sq.splits, rem = sq.tiles % sq.splits;
    t0 = split * base + min(split, rem);
    t1 = t0 + base + (split < rem ? 1 : 0);
    rows_here = min(kRowsPerGroup, sq.rows - rgi * kRowsPerGroup);
  }
  const int nt = t1 - t0;
  const bool row_mode = rows_here > 128;
  const int L = sq.L, T = sq.T;
  const bool need_anc = active && t1 * kTileKeys > L;


  const int kslots = row_mode ? 2 : 3;
  const int klead = row_mode ? 1 : 2;
  // Full barrier of K (is_v 0) or V (is_v 1) tile n and the parity of its
  // phase.  In key mode the groups take alternate tiles and share three-slot
  // rings, so each slot has one full barrier per group: a group then waits
  // on every phase of its barriers in order and never tests a barrier two
  // phases short of the tile it wants (the parity test would pass on the
  // wrong phase).
  auto full_bar = [&](int is_v, int n) -> int {
    const int base = is_v ? kVFull : kKFull;
    if (row_mode) return base + (is_v ? n % 3 : n % kslots);
    return base + n % 3 + 3 * (n & 1);
  };
  auto full_par = [&](int is_v, int n) -> uint32_t {
    if (row_mode) return (uint32_t)((is_v ? n / 3 : n / kslots) & 1);
    return (uint32_t)((n / 6) & 1);
  };
  auto kslot_addr = [&](int s) -> uint32_t { return s < 2 ? sK + s * TB : sQ + TB; };
  auto vslot_addr = [&](int s) -> uint32_t { return sV + s * TB; };
  // tiles of group g: row mode every tile, key mode every other tile
  auto ntiles = [&](int g) { return row_mode ? nt : (nt - g + 1) / 2; };
  auto tile_of = [&](int g, int j) { return row_mode ? j : 2 * j + g; };

  if (warp < 4) {
    if (!(active && nt > 0)) {
    } else if (warp == 0) {
      // ------------------------------------------------------------ loader
      const int P = a.plan.page_size;
      const int npg = kTileKeys / P;
      const int nops = npg;                       // TMA boxes (one per page) per tile
      const int32_t* ptab = a.page_table + (int64_t)p.b * a.plan.max_pages;
      // K and V are read once: evict-first, so that the stream leaves the
      // split outputs and chunk masses the finish kernel reads in L2
      const uint64_t kv_policy = l2_evict_first();
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        const int nq = row_mode ? 2 : 1;
        mbar_arrive_expect_tx(bar(kQFull), nq * TB);
        for (int qt = 0; qt < nq; ++qt) {
          const int j0 = (rgi * kRowsPerGroup + qt * 128) / G;
          for (int hf = 0; hf < NH; ++hf)
            tma_load_3d(sQ + qt * TB + hf * kHalfBytes, &tm_q, bar(kQFull), hf * 64, kvh * G,
                        sq.node0 + j0);
        }
      }
      // one tile of K (is_v = 0) or V (is_v = 1) into its ring slot
      auto load_tile = [&](int n, int is_v) -> bool {
        const int t = t0 + n;
        const int nslots = is_v ? 3 : kslots;
        const int slot = n % nslots;
        const int use = n / nslots;
        const uint32_t full = bar(full_bar(is_v, n));
        const uint32_t empty = bar((is_v ? kVEmpty : kKEmpty) + slot);
        const uint32_t dst = is_v ? vslot_addr(slot) : kslot_addr(slot);
        const int slot0 = t * kTileKeys;
        const int valid_end = L + T;           // slots below this hold real keys
        // Every page of the tile arrives by TMA except a page that holds the
        // sequence end (partially valid), which is copied with plain loads
        // so that its slots past the end read as zero.  Pages wholly past the
        // end get an out-of-range page coordinate: TMA fills them with zeros.
        int pg = 0;
        bool lane_tma = false;
        if (lane < nops) {
          const int ps = slot0 + lane * P;
          if (ps + P <= valid_end) {
            pg = __ldg(ptab + ps / P);
            if (pg < 0 || pg >= a.num_pages) {
              flag(a.plan.status, DS_DEV_BAD_PAGE);
              pg = a.num_pages;
            }
            lane_tma = true;
          } else if (ps >= valid_end) {
            pg = a.num_pages;
            lane_tma = true;
          }
        }
        const uint32_t tma_lanes = __ballot_sync(0xffffffffu, lane_tma);
        const bool partial = __popc(tma_lanes) != nops;
        if (lane == 0) ctrl->where[0] = 10000 + (is_v ? kVEmpty : kKEmpty) * 100 + n;
        if (!__all_sync(0xffffffffu, mbar_wait(empty, (use & 1) ^ 1, abort_flag, diag,
                                                10000 + (is_v ? kVEmpty : kKEmpty) * 100 + n)))
          return false;
        if (lane == 0) {
          if (partial)
            mbar_expect_tx(full, __popc(tma_lanes) * P * D * 2);
          else
            mbar_arrive_expect_tx(full, TB);
        }
        __syncwarp();
        if (lane_tma) {
          // coordinates (column, row in group, column half, row group, page);
          // the map folds the kv head into the half axis (NHD) or the page
          // axis (HND)
          const uint32_t d = dst + lane * P * D * 2;
          const CUtensorMap* m = is_v ? &tm_v : &tm_k;
          if (hnd)
            tma_load_5d_hint(d, m, full, 0, 0, 0, 0, pg * a.plan.num_kv_heads + kvh, kv_policy);
          else
            tma_load_5d_hint(d, m, full, 0, 0, kvh * NH, 0, pg, kv_policy);
        }
        if (partial) {
          // the one page with ps < valid_end < ps + P: plain 16-byte loads,
          // zeros past the end, written in the 128-byte swizzled layout
          const int pidx = (valid_end - slot0) / P;        // page index in the tile
          const int ps = slot0 + pidx * P;
          int pgi = __ldg(ptab + ps / P);
          const bool pg_ok = pgi >= 0 && pgi < a.num_pages;
          if (!pg_ok && lane == 0) flag(a.plan.status, DS_DEV_BAD_PAGE);
          const __nv_bfloat16* src = is_v ? a.v : a.k;
          constexpr int VPR = D / 8;                         // 16-byte chunks per row
          const int nelem = P * VPR;
          for (int base = 0; base < nelem; base += 32 * 8) {
            uint4 x[8];                                      // 8 loads in flight per lane
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              const int e = base + lane + 32 * r;
              x[r] = make_uint4(0, 0, 0, 0);
              if (e < nelem) {
                const int row = e / VPR, c = e % VPR;
                if (pg_ok && ps + row < valid_end) {
                  const int64_t off = (int64_t)pgi * a.page_stride +
                                      (int64_t)row * a.tok_stride +
                                      (int64_t)kvh * a.head_stride + c * 8;
                  x[r] = __ldg(reinterpret_cast<const uint4*>(src + off));
                }
              }
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              const int e = base + lane + 32 * r;
              if (e < nelem) {
                const int kk = pidx * P + e / VPR, c = e % VPR;
                const int hf = c >> 3, c8 = c & 7;
                const uint32_t d = dst + (kk >> 3) * Cfg<D>::RG + hf * 1024 + (kk & 7) * 128 +
                                   ((c8 ^ (kk & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(d), "r"(x[r].x),
                             "r"(x[r].y), "r"(x[r].z), "r"(x[r].w)
                             : "memory");
              }
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full);
        }
        return true;
      };
      bool ok = true;
      int nk = 0, nv = 0;   // tiles issued
      for (int n = 0; ok && n < klead && n < nt; ++n) ok = load_tile(n, 0), nk += ok;
      for (int n = 0; ok && n < nt; ++n) {
        ok = load_tile(n, 1);
        nv += ok;
        if (ok && n + klead < nt) ok = load_tile(n + klead, 0), nk += ok;
      }
      if (lane == 0) ctrl->where[0] = ok ? 19999 : 19998;
      // copies still in flight must land before the CTA can exit
      if (!ok && lane == 0) {
        for (int n = max(0, nk - kslots); n < nk; ++n)
          drain_wait(bar(full_bar(0, n)), full_par(0, n));
        for (int n = max(0, nv - 3); n < nv; ++n)
          drain_wait(bar(full_bar(1, n)), full_par(1, n));
      }
    } else if (warp == 1) {
      // ---------------------------------------------------- ancestor masks
      // Only the split that holds the tree's keys needs them, and only for
      // its last tile(s): they are formed here, beside the loader, and the
      // softmax warps wait for them (kAnc) just before the first unit that
      // holds tree keys.
      if (need_anc) {
        // ancestor masks of all nodes of this tree, by pointer doubling
        for (int j = lane; j < T; j += 32) ctrl->parents[j] = __ldg(a.parents + sq.node0 + j);
        __syncwarp();
        uint64_t m[2] = {0, 0};
        int up[2] = {-1, -1};
        for (int k = 0; k < 2; ++k) {
          const int j = lane + 32 * k;
          if (j < T) {
            int pj = ctrl->parents[j];
            bool ok = (j == 0) ? (pj == -1) : (pj >= 0 && pj < j);
            if (!ok) {
              flag(a.plan.status, DS_DEV_BAD_TREE);
              pj = -1;
            }
            m[k] = (1ull << j) | (pj >= 0 ? (1ull << pj) : 0ull);
            up[k] = pj;
            ctrl->anc[j] = m[k];
            ctrl->parents[j] = pj;   // sanitised jump pointer
          }
        }
        __syncwarp();
        for (int round = 0; round < 6; ++round) {
          uint64_t add[2] = {0, 0};
          int nup[2] = {-1, -1};
          for (int k = 0; k < 2; ++k) {
            const int j = lane + 32 * k;
            if (j < T && up[k] >= 0) {
              add[k] = ctrl->anc[up[k]];
              nup[k] = ctrl->parents[up[k]];
            }
          }
          __syncwarp();
          for (int k = 0; k < 2; ++k) {
            const int j = lane + 32 * k;
            if (j < T) {
              m[k] |= add[k];
              up[k] = nup[k];
              ctrl->anc[j] = m[k];
              ctrl->parents[j] = nup[k];
            }
          }
          __syncwarp();
        }
        mbar_arrive(bar(kAnc));
      }
    } else if (warp == 2 || warp == 3) {
      // ------------------------------------------------------ MMA issuers
      // One issuing thread per softmax group (warp 2: group 0, warp 3:
      // group 1).  A thread that has issued tcgen05.mma pays for any later
      // shared-memory access of its own with the time its queued MMAs need
      // to drain, so each group's MMAs come from a thread that only waits
      // on that group's P, at a point where its own MMAs have long
      // completed; the two groups never hold each other up.
      const int g = warp - 2;
      if (lane == 0) {
        constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 64, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
        // Descriptor bases computed once; each MMA only adds a compile-time
        // offset to the 14-bit start-address field (addresses stay below
        // 256 KB, so the add never carries into the neighbouring fields).
        const uint64_t qd0 = sdesc_sw128(sQ, 16, 1024);
        const uint64_t qb = (row_mode && g == 1) ? qd0 + (TB >> 4) : qd0;   // this group's Q
        constexpr uint32_t RG = Cfg<D>::RG;
        // K: K-major, 8-row groups RG bytes apart.  V: MN-major, the two
        // 64-column halves 1 KB apart (LBO), 8-key groups RG apart (SBO).
        const uint64_t kd0 = sdesc_sw128(sK, 16, RG);
        const uint64_t kd2 = sdesc_sw128(sQ + TB, 16, RG);        // K slot 2 (key mode)
        const uint64_t vd0 = sdesc_sw128(sV, 1024, RG);
        const uint32_t tG = tmem + (uint32_t)(256 * g);
        // users of each K and V tile: both groups in row mode, one in key
        // mode (which then releases the slot with two commits)
        const int rel = row_mode ? 1 : 2;
        auto kslot_of = [&](int t) { return row_mode ? (t & 1) : (t % 3); };
        // half slot h (64 columns at tG + 64 h) holds S, then P in place,
        // of keys 64 h .. 64 h + 63 of the group's current tile; O at
        // tG + 128.  S of a half slot's next tile is issued right after the
        // P V that reads the slot (the pipe runs in order), so the group's
        // next half is ready while it still works on the other half.
        auto qk = [&](int t, int h) {
          const int ks = kslot_of(t);
          const uint64_t kb = (ks < 2 ? kd0 + (uint64_t)(ks * (TB >> 4)) : kd2) +
                              (uint64_t)(h * ((8 * RG) >> 4));
          const uint32_t d = tG + (uint32_t)(64 * h);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t qoff = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
            const uint32_t koff = ((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
            mma_ss(d, qb + qoff, kb + koff, idesc_qk, kk > 0);
          }
        };
        // O += P(half h) V(keys 64 h .. 64 h + 63)
        auto pv = [&](int t, int h, bool acc) {
          const uint64_t vb = vd0 + (uint64_t)((t % 3) * (TB >> 4) + h * ((8 * RG) >> 4));
          const uint32_t pa = tG + (uint32_t)(64 * h);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tG + 128, pa + kk * 8, vb + (uint64_t)(kk * ((2 * RG) >> 4)), idesc_pv,
                   (acc || kk > 0) ? 1u : 0u);
        };
        const int wi = g == 0 ? 1 : 4;   // this issuer's slot in ctrl->where
        auto wait = [&](int b, uint32_t par, uint32_t tag) {
          ctrl->where[wi] = tag;
          return mbar_wait(bar(b), par, abort_flag, diag, tag);
        };
        auto wait_k = [&](int t) {
          return wait(full_bar(0, t), full_par(0, t), 20000 + kKFull * 100 + t);
        };
        auto wait_v = [&](int n) {
          return wait(full_bar(1, n), full_par(1, n), 20000 + kVFull * 100 + n);
        };
        const int my_nt = ntiles(g);
        bool ok = wait(kQFull, 0, 20000 + kQFull * 100);
        // prologue: S of both halves of the group's first tile
        if (ok && my_nt > 0) {
          const int t = tile_of(g, 0);
          if ((ok = wait_k(t))) {
            tc_fence_after();
            for (int h = 0; h < 2; ++h) {
              qk(t, h);
              mma_commit(bar(kSFull + 2 * g + h));
            }
            for (int r = 0; r < rel; ++r) mma_commit(bar(kKEmpty + kslot_of(t)));
          }
        }
        for (int j = 0; ok && j < my_nt; ++j) {
          const int n = tile_of(g, j);
          const bool more = j + 1 < my_nt;
          const int tn = more ? tile_of(g, j + 1) : 0;
          for (int h = 0; h < 2; ++h) {
            if (!(ok = wait(kPFull + 2 * g + h, j & 1,
                            20000 + (kPFull + 2 * g + h) * 100 + 2 * j + h)))
              break;
            if (h == 0 && !(ok = wait_v(n))) break;
            tc_fence_after();
            pv(n, h, j > 0 || h > 0);
            mma_commit(bar(kORdy + g));
            if (more) {
              // the next tile's K is waited for only now, so that a late K
              // copy does not hold back this half's P V
              if (h == 0) {
                if (!(ok = wait_k(tn))) break;
                tc_fence_after();
              }
              qk(tn, h);
              mma_commit(bar(kSFull + 2 * g + h));
              if (h == 1)
                for (int r = 0; r < rel; ++r) mma_commit(bar(kKEmpty + kslot_of(tn)));
            }
            if (h == 1)
              for (int r = 0; r < rel; ++r) mma_commit(bar(kVEmpty + n % 3));
          }
        }
        // all issued MMAs complete -> epilogue (also on the abort path, so
        // that nothing is in flight when tensor memory is freed)
        if (ok) ctrl->where[wi] = 29999;
        mma_commit(bar(kOFinal + g));
      }
    }
  } else {
    if (active && nt > 0) {
      // ------------------------------------------------------------ softmax
      const int g = (warp - 4) >> 2;                 // softmax group
      const int q4 = warp & 3;                       // TMEM lane quarter
      const int lrow = q4 * 32 + lane;               // row inside the Q tile
      const int grow_local = row_mode ? g * 128 + lrow : lrow;
      const bool row_ok = grow_local < rows_here;
      const int grow = rgi * kRowsPerGroup + grow_local;
      const int jn = grow / G;
      uint64_t anc = 0ull;          // read at the first unit with tree keys
      bool anc_ready = !need_anc;
      const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
      const uint32_t tG = tmem + lane_addr + 256 * g;
      const uint32_t tO = tG + 128;
      const float c2 = a.scale_log2;
      const int C = a.plan.chunk_size;
      const int cshift = __ffs(C) - 1;               // C is a power of two >= 16
      const int n_ch = (L + C - 1) / C;
      float* clse_row = a.clse +
                        (((int64_t)p.b * a.plan.num_kv_heads + kvh) * a.plan.rg_max + rgi) *
                            a.plan.max_chunks * kRowsPerGroup +
                        grow_local;
      float m2 = -CUDART_INF_F, l = 0.f, cs = 0.f;
      bool ok = true;
      const int my_nt = ntiles(g);
      for (int j = 0; ok && j < my_nt; ++j) {
        const int n = tile_of(g, j);
        const int tile_slot0 = (t0 + n) * kTileKeys;
        for (int hb = 0; hb < 2; ++hb) {
          const int u = 2 * j + hb;
          if (lrow == 0) ctrl->where[2 + g] = 30000 + (kSFull + 2 * g + hb) * 100 + j;
          ok = __all_sync(0xffffffffu, mbar_wait(bar(kSFull + 2 * g + hb), j & 1, abort_flag,
                                                 diag, 30000 + (kSFull + 2 * g + hb) * 100 + j));
          if (!ok) break;
          tc_fence_after();
          const uint32_t tS = tG + 64 * hb;     // scores of keys 64 hb .. 64 hb + 63
          const uint32_t tP = tS;               // their P (bf16 pairs), in place
          const int unit_slot0 = tile_slot0 + 64 * hb;
          float alpha;
          bool rescale;
          if (unit_slot0 + 64 <= L) {
            softmax_unit<false>(tS, tP, ~0u, ~0u, ~0u, ~0u, c2, u == 0, m2, l, cs, alpha,
                                rescale, tile_slot0, 4 * hb, cshift, n_ch, row_ok, clse_row);
          } else {
            if (!anc_ready) {
              if (lrow == 0) ctrl->where[2 + g] = 30000 + kAnc * 100;
              ok = __all_sync(0xffffffffu, mbar_wait(bar(kAnc), 0, abort_flag, diag,
                                                     30000 + kAnc * 100));
              if (!ok) break;
              anc = (row_ok && jn < T) ? ctrl->anc[jn] : 0ull;
              anc_ready = true;
            }
            // column c is visible iff c < L - unit_slot0 (context) or it is
            // tree slot i = c - (L - unit_slot0) with bit i of the row's
            // ancestor mask set
            const int off = L - unit_slot0;
            const uint64_t ctx = off >= 64 ? ~0ull : (off <= 0 ? 0ull : ((1ull << off) - 1));
            const uint64_t tr = off >= 0 ? (off >= 64 ? 0ull : (anc << off))
                                         : (-off >= 64 ? 0ull : (anc >> (-off)));
            const uint64_t vis = ctx | tr;
            softmax_unit<true>(tS, tP, (uint32_t)vis, (uint32_t)(vis >> 32), (uint32_t)ctx,
                               (uint32_t)(ctx >> 32), c2, u == 0, m2, l, cs, alpha, rescale,
                               tile_slot0, 4 * hb, cshift, n_ch, row_ok, clse_row);
          }
          if (rescale) {
            // O must hold the sum over all earlier halves: wait for the
            // previous half's P V (the one before it completed before this
            // half's S, which was issued after it)
            if (lrow == 0) ctrl->where[2 + g] = 30000 + (kORdy + g) * 100 + u;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kORdy + g), (u - 1) & 1, abort_flag,
                                                   diag, 30000 + (kORdy + g) * 100 + u));
            if (ok) {
              tc_fence_after();
#pragma unroll 1
              for (int c4 = 0; c4 < D / 32; ++c4) {
                uint32_t r[32];
                tmem_ld32(tO + c4 * 32, r);
                tmem_ld_wait(r);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                tmem_st32(tO + c4 * 32, r);
              }
            }
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(kPFull + 2 * g + hb));
          if (!ok) break;
        }
      }
      // ------------------------------------------------------------ epilogue
      // key mode merges the groups through shared memory that the V ring
      // uses, so there both groups' MMAs must be complete (and with them
      // every V load); row mode needs only the group's own
      if (lrow == 0) ctrl->where[2 + g] = 30000 + (kOFinal + g) * 100;
      if (ok)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kOFinal + g), 0, abort_flag, diag,
                                               30000 + (kOFinal + g) * 100));
      if (ok && !row_mode)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kOFinal + 1 - g), 0, abort_flag, diag,
                                               30000 + (kOFinal + 1 - g) * 100));
      else __syncwarp();
      if (ok) tc_fence_after();
      const int nt1 = row_mode ? 0 : ntiles(1);    // tiles of group 1 in key mode
      // staging (4 warps x 4 KB, within a Q tile even at head_dim 64): the
      // group's own Q tile, idle once its MMAs are complete (key mode: Q
      // tile 0, idle once both groups' are)
      float* stage = reinterpret_cast<float*>(smem + (row_mode ? g * TB : 0)) +
                     q4 * 32 * kStageStride;
      const int warp_row0 = grow_local - lane;       // first row of this warp
      // the split outputs are kept at the precision of the final output
      const int64_t orow = ((int64_t)blockIdx.x * kRowsPerGroup + warp_row0) * D;
      void* op_warp = a.out_f32 ? static_cast<void*>(a.o_part + orow)
                                : static_cast<void*>(
                                      reinterpret_cast<__nv_bfloat16*>(a.o_part) + orow);
      write_row_output<D>(row_mode, g, ok, nt1, tO, lrow, rows_here - warp_row0, m2, l,
                          merge_buf, m1buf, l1buf, stage, !a.out_f32, op_warp,
                          a.lse_part + (int64_t)blockIdx.x * kRowsPerGroup + grow_local);
    }
  }

  // --------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    flag(a.plan.status, DS_DEV_TIMEOUT);
    if (diag[1] == blockIdx.x)
      for (int i = 0; i < 5; ++i) diag[2 + i] = ctrl->where[i];
  }
  if (active && nt > 0) {
    // The last split of a (sequence, kv head, row group) to finish forms
    // the rows' final log2-sum-exp from every split's, and records where
    // the row group's splits are, so that the finish kernel can merge
    // outputs and normalise chunk masses independently.  Every split counts
    // (a timed-out one too), and the last resets the counter to zero for
    // the next call.
    const int64_t cidx = ((int64_t)p.b * a.plan.num_kv_heads + kvh) * a.plan.rg_max + rgi;
    const int64_t base = (int64_t)sq.item_base + (kvh * sq.rg + rgi) * sq.splits;
    if (threadIdx.x == 0) {
      __threadfence();            // this split's outputs before its arrival
      const uint32_t prev = atomicAdd(a.counters + cidx, 1u);
      const int last = prev + 1 == (uint32_t)sq.splits;
      if (last) {
        a.counters[cidx] = 0u;
        a.gdesc[cidx] = make_int4((int)base, sq.splits, 0, 0);
        __threadfence();          // the other splits' outputs before reading them
      }
      ctrl->last = last;
    }
    __syncthreads();
    if (ctrl->last)
      for (int r = threadIdx.x; r < rows_here; r += kThreads)
        a.row_lse[cidx * kRowsPerGroup + r] =
            row_lse_from_splits(a.lse_part + base * kRowsPerGroup + r, sq.splits);
  }
  if (warp == 1) {
    if (active && nt > 0 && lane == 0) {
      drain_wait(bar(kOFinal), 0);
      drain_wait(bar(kOFinal + 1), 0);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace tc

// ---------------------------------------------------------------------------
// host side

namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  }
  return fn;
}

bool encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_tc(const VerifyKArgs& k, const ds_verify_args& a, const VerifyLayout& L,
                      cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  const int G = L.group;
  const cuuint64_t P = a.page_size, H = a.num_kv_heads, NP = a.num_pages;
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.num_q_heads, (cuuint64_t)a.n_nodes};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.num_q_heads * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(128 / G)};
    if (!encode(&tq, a.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  // K and V: one box is one page of one kv head, all columns, landing as
  // [row group of 8][column half][8 rows x 128 bytes].  Axes: column (64),
  // row in group (8), column half, row group (P / 8), page.  NHD
  // [pages, P, H, D]: the kv head is folded into the half axis (halves of
  // consecutive heads are 128 bytes apart).  HND [pages, H, P, D]: the kv
  // head is folded into the page axis (coordinate page * H + head).
  const bool hnd = a.kv_layout == DS_KV_HND;
  constexpr cuuint64_t NH = D / 64;
  cuuint64_t dims[5], strides[4];
  const cuuint32_t box[5] = {64, 8, (cuuint32_t)NH, (cuuint32_t)(P / 8), 1};
  if (!hnd) {
    const cuuint64_t row = H * D * 2;
    const cuuint64_t d[5] = {64, 8, NH * H, P / 8, NP};
    const cuuint64_t s[4] = {row, 128, 8 * row, P * row};
    for (int i = 0; i < 5; ++i) dims[i] = d[i];
    for (int i = 0; i < 4; ++i) strides[i] = s[i];
  } else {
    const cuuint64_t row = D * 2;
    const cuuint64_t d[5] = {64, 8, NH, P / 8, H * NP};
    const cuuint64_t s[4] = {row, 128, 8 * row, P * row};
    for (int i = 0; i < 5; ++i) dims[i] = d[i];
    for (int i = 0; i < 4; ++i) strides[i] = s[i];
  }
  if (!encode(&tk, a.k_cache, 5, dims, strides, box)) return cudaErrorInvalidValue;
  if (!encode(&tv, a.v_cache, 5, dims, strides, box)) return cudaErrorInvalidValue;
  const size_t smem = tc::Cfg<D>::smem;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(tc::verify_split_tc<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_dependent(tc::verify_split_tc<D>, dim3(L.max_items), dim3(tc::kThreads), smem,
                          stream, tq, tk, tv, k, hnd ? 1 : 0);
}

}  // namespace

cudaError_t launch_split_tc(const VerifyKArgs& k, const ds_verify_args& a,
                            const VerifyLayout& L, cudaStream_t stream) {
  if (a.head_dim == 128) return launch_tc<128>(k, a, L, stream);
  return launch_tc<64>(k, a, L, stream);
}

}  // namespace ds
