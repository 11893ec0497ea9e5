// C ABI of the tree-verify library: host-side validation, workspace layouts
// and dispatch to the kernel launchers.  Every refusal happens here, before
// any work is enqueued, and names the offending argument.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "ds.h"
#include "internal.h"

namespace {

thread_local std::string g_err;

ds_status fail(ds_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

ds_status ok() {
  g_err.clear();
  return DS_OK;
}

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ds_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int device_sms(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  return 0;
}

#define REQUIRE(cond, st, ...) \
  do {                         \
    if (!(cond)) return fail(st, __VA_ARGS__); \
  } while (0)

// ---------------------------------------------------------------------------
ds_status check_verify_sizes(const ds_verify_args* a) {
  REQUIRE(a, DS_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->batch >= 1, DS_ERR_INVALID_ARG, "batch must be >= 1 (got %d)", a->batch);
  REQUIRE(a->n_nodes >= 0, DS_ERR_INVALID_ARG, "n_nodes must be >= 0 (got %d)", a->n_nodes);
  REQUIRE(a->num_kv_heads >= 1, DS_ERR_INVALID_ARG, "num_kv_heads must be >= 1");
  REQUIRE(a->num_q_heads >= a->num_kv_heads && a->num_q_heads % a->num_kv_heads == 0,
          DS_ERR_UNSUPPORTED,
          "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
          a->num_q_heads, a->num_kv_heads);
  const int G = a->num_q_heads / a->num_kv_heads;
  REQUIRE(pow2(G) && G <= 16, DS_ERR_UNSUPPORTED,
          "group size num_q_heads/num_kv_heads = %d: only powers of two up to 16", G);
  REQUIRE(a->head_dim == 64 || a->head_dim == 128, DS_ERR_UNSUPPORTED,
          "head_dim %d: only 64 and 128 are supported", a->head_dim);
  REQUIRE(a->page_size == 16 || a->page_size == 32 || a->page_size == 64 ||
              a->page_size == 128,
          DS_ERR_UNSUPPORTED, "page_size %d: only 16, 32, 64 or 128", a->page_size);
  REQUIRE(a->chunk_size > 0 && pow2(a->chunk_size) && a->chunk_size <= 128 &&
              a->chunk_size % a->page_size == 0,
          DS_ERR_UNSUPPORTED,
          "chunk_size %d: must be a power of two, a multiple of page_size (%d), <= 128",
          a->chunk_size, a->page_size);
  REQUIRE(a->num_pages >= 1, DS_ERR_INVALID_ARG, "num_pages must be >= 1");
  REQUIRE(a->max_pages >= 1, DS_ERR_INVALID_ARG, "max_pages must be >= 1");
  REQUIRE(a->max_chunks >= 0, DS_ERR_INVALID_ARG, "max_chunks must be >= 0");
  REQUIRE(a->kv_layout == DS_KV_NHD || a->kv_layout == DS_KV_HND, DS_ERR_INVALID_ARG,
          "kv_layout %d is not a ds_kv_layout", a->kv_layout);
  REQUIRE(a->out_dtype == DS_OUT_BF16 || a->out_dtype == DS_OUT_F32, DS_ERR_INVALID_ARG,
          "out_dtype %d is not a ds_out_dtype", a->out_dtype);
  REQUIRE(a->accumulate_scores == 0 || a->accumulate_scores == 1, DS_ERR_INVALID_ARG,
          "accumulate_scores must be 0 or 1");
  REQUIRE(std::isfinite(a->scale) && a->scale >= 0.f, DS_ERR_INVALID_ARG,
          "scale must be finite and >= 0 (0 selects 1/sqrt(head_dim))");
  REQUIRE(a->num_sms >= 0, DS_ERR_INVALID_ARG, "num_sms must be >= 0");
  const int64_t cache_elems = (int64_t)a->num_pages * a->page_size * a->num_kv_heads *
                              a->head_dim;
  REQUIRE(cache_elems < (int64_t)1 << 40, DS_ERR_UNSUPPORTED, "cache too large");
  // the HND tensor map addresses (page, kv head) as one coordinate
  REQUIRE((int64_t)(a->num_pages + 1) * a->num_kv_heads < ((int64_t)1 << 31),
          DS_ERR_UNSUPPORTED, "num_pages * num_kv_heads must stay below 2^31");
  return DS_OK;
}

}  // namespace

namespace ds {

VerifyLayout verify_layout(const ds_verify_args& a, int num_sms) {
  VerifyLayout L;
  L.group = a.num_q_heads / a.num_kv_heads;
  L.rg_max = (DS_MAX_TREE_NODES * L.group + kRowsPerItem - 1) / kRowsPerItem;
  L.target_ctas = num_sms;
  // A batch of sequences of different lengths can round its splits badly in
  // one wave of num_sms CTAs; the plan may then use two (see plan_refit), so
  // the grid and the split outputs are sized for it.  A single sequence's
  // row groups all have the same length and never need it.
  L.wave_ctas = a.batch > 1 ? 2 * num_sms : 0;
  L.max_items = (L.wave_ctas > 0 ? L.wave_ctas : num_sms) + a.batch * a.num_kv_heads * L.rg_max;
  size_t off = kStatusBytes;
  L.counters = off;
  off = align_up(off + (size_t)a.batch * a.num_kv_heads * L.rg_max * sizeof(uint32_t));
  L.gdesc = off;
  off = align_up(off + (size_t)a.batch * a.num_kv_heads * L.rg_max * sizeof(int32_t) * 4);
  L.o_part = off;
  off = align_up(off + (size_t)L.max_items * kRowsPerItem * a.head_dim * sizeof(float));
  L.lse_part = off;
  off = align_up(off + (size_t)L.max_items * kRowsPerItem * sizeof(float));
  L.clse = off;
  off = align_up(off + (size_t)a.batch * a.num_kv_heads * L.rg_max * a.max_chunks * kRowsPerItem *
                           sizeof(float));
  L.row_lse = off;
  off = align_up(off + (size_t)a.batch * a.num_kv_heads * L.rg_max * kRowsPerItem * sizeof(float));
  L.total = off;
  return L;
}

AcceptLayout accept_layout(const ds_accept_args& a) {
  AcceptLayout L;
  L.node_stats = kStatusBytes;
  L.total = align_up(kStatusBytes + (size_t)(a.n_nodes > 0 ? a.n_nodes : 0) * sizeof(NodeStats));
  return L;
}

ds_status set_last_error(ds_status st, const char* msg) {
  g_err = msg;
  return st;
}

}  // namespace ds

extern "C" {

const char* ds_last_error(void) { return g_err.c_str(); }

int32_t ds_abi_version(void) { return DS_ABI_VERSION; }

int64_t ds_struct_size(int32_t which) {
  switch (which) {
    case 0: return (int64_t)sizeof(ds_verify_args);
    case 1: return (int64_t)sizeof(ds_gather_args);
    case 2: return (int64_t)sizeof(ds_accept_args);
    case 3: return (int64_t)sizeof(ds_commit_args);
    case 4: return (int64_t)sizeof(ds_append_args);
    default: return -1;
  }
}

ds_status ds_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  REQUIRE(workspace, DS_ERR_WORKSPACE, "workspace is NULL");
  REQUIRE(workspace_bytes >= ds::kStatusBytes, DS_ERR_WORKSPACE,
          "workspace_bytes %zu below the %zu-byte status region", workspace_bytes,
          ds::kStatusBytes);
  cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ds_workspace_init");
  return ok();
}

ds_status ds_device_status(const void* workspace, uint32_t* flags, void* stream) {
  REQUIRE(workspace, DS_ERR_WORKSPACE, "workspace is NULL");
  REQUIRE(flags, DS_ERR_INVALID_ARG, "flags is NULL");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ds_device_status: stream synchronize");
  e = cudaMemcpy(flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "ds_device_status: copy");
  return ok();
}

// ---------------------------------------------------------------------------
void ds_verify_args_default(ds_verify_args* a) {
  if (!a) return;
  std::memset(a, 0, sizeof(*a));
  a->kv_layout = DS_KV_NHD;
  a->out_dtype = DS_OUT_BF16;
}

ds_status ds_verify_attn_workspace_size(const ds_verify_args* a, size_t* bytes) {
  ds_status st = check_verify_sizes(a);
  if (st != DS_OK) return st;
  REQUIRE(bytes, DS_ERR_INVALID_ARG, "bytes is NULL");
  int sms = a->num_sms;
  if (sms == 0 && device_sms(&sms) != 0)
    return fail(DS_ERR_CUDA, "num_sms is 0 and the device SM count is unavailable");
  *bytes = ds::verify_layout(*a, sms).total;
  return ok();
}

ds_status ds_verify_attn(const ds_verify_args* a, void* stream) {
  ds_status st = check_verify_sizes(a);
  if (st != DS_OK) return st;
  REQUIRE(a->q || a->n_nodes == 0, DS_ERR_INVALID_ARG, "q is NULL");
  REQUIRE(a->k_cache, DS_ERR_INVALID_ARG, "k_cache is NULL");
  REQUIRE(a->v_cache, DS_ERR_INVALID_ARG, "v_cache is NULL");
  REQUIRE(a->page_table, DS_ERR_INVALID_ARG, "page_table is NULL");
  REQUIRE(a->ctx_lens, DS_ERR_INVALID_ARG, "ctx_lens is NULL");
  REQUIRE(a->tree_offsets, DS_ERR_INVALID_ARG, "tree_offsets is NULL");
  REQUIRE(a->parents || a->n_nodes == 0, DS_ERR_INVALID_ARG, "parents is NULL");
  REQUIRE(a->out || a->n_nodes == 0, DS_ERR_INVALID_ARG, "out is NULL");
  REQUIRE(a->chunk_scores || a->max_chunks == 0, DS_ERR_INVALID_ARG,
          "chunk_scores is NULL");
  REQUIRE(aligned16(a->q) && aligned16(a->k_cache) && aligned16(a->v_cache) &&
              aligned16(a->out),
          DS_ERR_INVALID_ARG, "q, k_cache, v_cache and out must be 16-byte aligned");
  REQUIRE(a->workspace, DS_ERR_WORKSPACE, "workspace is NULL");
  REQUIRE((reinterpret_cast<uintptr_t>(a->workspace) & (ds::kAlign - 1)) == 0,
          DS_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  int sms = a->num_sms;
  if (sms == 0 && device_sms(&sms) != 0)
    return fail(DS_ERR_CUDA, "num_sms is 0 and the device SM count is unavailable");
  const ds::VerifyLayout L = ds::verify_layout(*a, sms);
  REQUIRE(a->workspace_bytes >= L.total, DS_ERR_WORKSPACE,
          "workspace_bytes %zu < required %zu", a->workspace_bytes, L.total);
  if (a->n_nodes == 0) return ok();
  cudaError_t e = ds::launch_verify(*a, L, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ds_verify_attn launch");
  return ok();
}

// ---------------------------------------------------------------------------
void ds_gather_args_default(ds_gather_args* a) {
  if (!a) return;
  std::memset(a, 0, sizeof(*a));
  a->kv_layout = DS_KV_NHD;
}

static ds_status check_gather(const ds_gather_args* a) {
  REQUIRE(a, DS_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->batch >= 1, DS_ERR_INVALID_ARG, "batch must be >= 1 (got %d)", a->batch);
  REQUIRE(a->num_kv_heads >= 1, DS_ERR_INVALID_ARG, "num_kv_heads must be >= 1");
  REQUIRE(a->head_dim == 64 || a->head_dim == 128, DS_ERR_UNSUPPORTED,
          "head_dim %d: only 64 and 128 are supported", a->head_dim);
  REQUIRE(a->page_size >= 1, DS_ERR_INVALID_ARG, "page_size must be >= 1");
  REQUIRE(a->chunk_size >= 1 && a->chunk_size % a->page_size == 0, DS_ERR_UNSUPPORTED,
          "chunk_size %d must be a positive multiple of page_size %d", a->chunk_size,
          a->page_size);
  REQUIRE(a->top_k >= 0, DS_ERR_INVALID_ARG, "top_k must be >= 0");
  REQUIRE(a->window >= 0, DS_ERR_INVALID_ARG, "window must be >= 0");
  REQUIRE(a->max_chunks >= 0, DS_ERR_INVALID_ARG, "max_chunks must be >= 0");
  REQUIRE(a->num_pages >= 1 && a->max_pages >= 1, DS_ERR_INVALID_ARG,
          "num_pages and max_pages must be >= 1");
  REQUIRE(a->kv_layout == DS_KV_NHD || a->kv_layout == DS_KV_HND, DS_ERR_INVALID_ARG,
          "kv_layout %d is not a ds_kv_layout", a->kv_layout);
  REQUIRE(a->rope_base >= 0.f && a->rope_base < 3.0e38f, DS_ERR_INVALID_ARG,
          "rope_base must be 0 (no rotation) or a finite positive base");
  REQUIRE((int64_t)a->capacity >= (int64_t)a->top_k * a->chunk_size + a->window,
          DS_ERR_INVALID_ARG, "capacity %d < top_k*chunk_size + window = %lld",
          a->capacity, (long long)a->top_k * a->chunk_size + a->window);
  return DS_OK;
}

ds_status ds_chunk_topk_gather_workspace_size(const ds_gather_args* a, size_t* bytes) {
  ds_status st = check_gather(a);
  if (st != DS_OK) return st;
  REQUIRE(bytes, DS_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = ds::kStatusBytes;
  return ok();
}

ds_status ds_chunk_topk_gather(const ds_gather_args* a, void* stream) {
  ds_status st = check_gather(a);
  if (st != DS_OK) return st;
  REQUIRE(a->scores || a->max_chunks == 0, DS_ERR_INVALID_ARG, "scores is NULL");
  REQUIRE(a->ctx_lens, DS_ERR_INVALID_ARG, "ctx_lens is NULL");
  REQUIRE(a->src_k && a->src_v, DS_ERR_INVALID_ARG, "src_k/src_v is NULL");
  REQUIRE(a->page_table, DS_ERR_INVALID_ARG, "page_table is NULL");
  REQUIRE(a->out_k && a->out_v, DS_ERR_INVALID_ARG, "out_k/out_v is NULL");
  REQUIRE(a->out_positions, DS_ERR_INVALID_ARG, "out_positions is NULL");
  REQUIRE(a->out_len, DS_ERR_INVALID_ARG, "out_len is NULL");
  REQUIRE(a->out_chunk_ids || a->top_k == 0, DS_ERR_INVALID_ARG, "out_chunk_ids is NULL");
  REQUIRE(aligned16(a->src_k) && aligned16(a->src_v) && aligned16(a->out_k) &&
              aligned16(a->out_v),
          DS_ERR_INVALID_ARG, "src_k, src_v, out_k and out_v must be 16-byte aligned");
  REQUIRE(a->workspace && a->workspace_bytes >= ds::kStatusBytes, DS_ERR_WORKSPACE,
          "workspace must hold at least %zu bytes", ds::kStatusBytes);
  if (a->capacity == 0) return ok();
  cudaError_t e = ds::launch_topk_gather(*a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ds_chunk_topk_gather launch");
  return ok();
}

// ---------------------------------------------------------------------------
void ds_accept_args_default(ds_accept_args* a) {
  if (!a) return;
  std::memset(a, 0, sizeof(*a));
  a->mode = DS_ACCEPT_GREEDY;
}

static ds_status check_accept(const ds_accept_args* a) {
  REQUIRE(a, DS_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->mode == DS_ACCEPT_GREEDY || a->mode == DS_ACCEPT_REJECT, DS_ERR_INVALID_ARG,
          "mode %d is not a ds_accept_mode", a->mode);
  REQUIRE(a->batch >= 1, DS_ERR_INVALID_ARG, "batch must be >= 1 (got %d)", a->batch);
  REQUIRE(a->n_nodes >= 0, DS_ERR_INVALID_ARG, "n_nodes must be >= 0");
  REQUIRE(a->vocab >= 1, DS_ERR_INVALID_ARG, "vocab must be >= 1");
  return DS_OK;
}

ds_status ds_accept_workspace_size(const ds_accept_args* a, size_t* bytes) {
  ds_status st = check_accept(a);
  if (st != DS_OK) return st;
  REQUIRE(bytes, DS_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = ds::accept_layout(*a).total;
  return ok();
}

ds_status ds_accept(const ds_accept_args* a, void* stream) {
  ds_status st = check_accept(a);
  if (st != DS_OK) return st;
  REQUIRE(a->target_logits || a->n_nodes == 0, DS_ERR_INVALID_ARG, "target_logits is NULL");
  REQUIRE(a->draft_tokens || a->n_nodes == 0, DS_ERR_INVALID_ARG, "draft_tokens is NULL");
  REQUIRE(a->parents || a->n_nodes == 0, DS_ERR_INVALID_ARG, "parents is NULL");
  REQUIRE(a->tree_offsets, DS_ERR_INVALID_ARG, "tree_offsets is NULL");
  REQUIRE(a->out_path && a->out_n_accepted && a->out_bonus, DS_ERR_INVALID_ARG,
          "out_path/out_n_accepted/out_bonus is NULL");
  if (a->mode == DS_ACCEPT_REJECT) {
    REQUIRE(a->draft_logits || a->n_nodes == 0, DS_ERR_INVALID_ARG,
            "draft_logits is NULL in rejection mode");
    REQUIRE(a->uniforms || a->n_nodes == 0, DS_ERR_INVALID_ARG,
            "uniforms is NULL in rejection mode");
  }
  const ds::AcceptLayout L = ds::accept_layout(*a);
  REQUIRE(a->workspace, DS_ERR_WORKSPACE, "workspace is NULL");
  REQUIRE((reinterpret_cast<uintptr_t>(a->workspace) & (ds::kAlign - 1)) == 0,
          DS_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  REQUIRE(a->workspace_bytes >= L.total, DS_ERR_WORKSPACE,
          "workspace_bytes %zu < required %zu", a->workspace_bytes, L.total);
  cudaError_t e = ds::launch_accept(*a, L, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ds_accept launch");
  return ok();
}

// ---------------------------------------------------------------------------
void ds_commit_args_default(ds_commit_args* a) {
  if (!a) return;
  std::memset(a, 0, sizeof(*a));
  a->kv_layout = DS_KV_NHD;
}

ds_status ds_kv_commit(const ds_commit_args* a, void* stream) {
  REQUIRE(a, DS_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->num_layers >= 1 && a->num_layers <= DS_MAX_COMMIT_LAYERS, DS_ERR_UNSUPPORTED,
          "num_layers %d outside 1..%d", a->num_layers, DS_MAX_COMMIT_LAYERS);
  REQUIRE(a->k_caches && a->v_caches, DS_ERR_INVALID_ARG, "k_caches/v_caches is NULL");
  for (int l = 0; l < a->num_layers; ++l) {
    REQUIRE(a->k_caches[l] && a->v_caches[l], DS_ERR_INVALID_ARG,
            "k_caches[%d]/v_caches[%d] is NULL", l, l);
    REQUIRE(aligned16(a->k_caches[l]) && aligned16(a->v_caches[l]), DS_ERR_INVALID_ARG,
            "caches of layer %d must be 16-byte aligned", l);
  }
  REQUIRE(a->batch >= 1, DS_ERR_INVALID_ARG, "batch must be >= 1 (got %d)", a->batch);
  REQUIRE(a->num_kv_heads >= 1, DS_ERR_INVALID_ARG, "num_kv_heads must be >= 1");
  REQUIRE(a->head_dim == 64 || a->head_dim == 128, DS_ERR_UNSUPPORTED,
          "head_dim %d (64 or 128)", a->head_dim);
  REQUIRE(a->page_size == 16 || a->page_size == 32 || a->page_size == 64 ||
              a->page_size == 128,
          DS_ERR_UNSUPPORTED, "page_size %d (16, 32, 64 or 128)", a->page_size);
  REQUIRE(a->num_pages >= 1 && a->max_pages >= 1, DS_ERR_INVALID_ARG,
          "num_pages and max_pages must be >= 1");
  REQUIRE(a->kv_layout == DS_KV_NHD || a->kv_layout == DS_KV_HND, DS_ERR_INVALID_ARG,
          "kv_layout %d is not a ds_kv_layout", a->kv_layout);
  REQUIRE(a->page_table && a->ctx_lens && a->tree_offsets && a->path && a->n_accepted,
          DS_ERR_INVALID_ARG, "page_table/ctx_lens/tree_offsets/path/n_accepted is NULL");
  REQUIRE(a->new_ctx_lens, DS_ERR_INVALID_ARG, "new_ctx_lens is NULL");
  REQUIRE((const void*)a->new_ctx_lens != (const void*)a->ctx_lens, DS_ERR_INVALID_ARG,
          "new_ctx_lens must not alias ctx_lens");
  REQUIRE(a->workspace, DS_ERR_WORKSPACE, "workspace is NULL");
  REQUIRE(a->workspace_bytes >= ds::kStatusBytes, DS_ERR_WORKSPACE,
          "workspace_bytes %zu < %zu", a->workspace_bytes, ds::kStatusBytes);
  cudaError_t e = ds::launch_kv_commit(*a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ds_kv_commit launch");
  return ok();
}

// ---------------------------------------------------------------------------
void ds_append_args_default(ds_append_args* a) {
  if (!a) return;
  std::memset(a, 0, sizeof(*a));
  a->kv_layout = DS_KV_NHD;
}

ds_status ds_compact_append(const ds_append_args* a, void* stream) {
  REQUIRE(a, DS_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->batch >= 1, DS_ERR_INVALID_ARG, "batch must be >= 1 (got %d)", a->batch);
  REQUIRE(a->num_kv_heads >= 1, DS_ERR_INVALID_ARG, "num_kv_heads must be >= 1");
  REQUIRE(a->head_dim == 64 || a->head_dim == 128, DS_ERR_UNSUPPORTED,
          "head_dim %d (64 or 128)", a->head_dim);
  REQUIRE(a->page_size >= 1, DS_ERR_INVALID_ARG, "page_size must be >= 1");
  REQUIRE(a->num_pages >= 1 && a->max_pages >= 1, DS_ERR_INVALID_ARG,
          "num_pages and max_pages must be >= 1");
  REQUIRE(a->kv_layout == DS_KV_NHD || a->kv_layout == DS_KV_HND, DS_ERR_INVALID_ARG,
          "kv_layout %d is not a ds_kv_layout", a->kv_layout);
  REQUIRE(a->capacity >= 0, DS_ERR_INVALID_ARG, "capacity must be >= 0");
  REQUIRE(a->rope_base >= 0.f && a->rope_base < 3.0e38f, DS_ERR_INVALID_ARG,
          "rope_base must be 0 (no rotation) or a finite positive base");
  REQUIRE(a->src_k && a->src_v && a->page_table && a->from_lens && a->to_lens,
          DS_ERR_INVALID_ARG, "src_k/src_v/page_table/from_lens/to_lens is NULL");
  REQUIRE(a->out_k && a->out_v && a->out_positions && a->out_len, DS_ERR_INVALID_ARG,
          "out_k/out_v/out_positions/out_len is NULL");
  REQUIRE(aligned16(a->src_k) && aligned16(a->src_v) && aligned16(a->out_k) &&
              aligned16(a->out_v),
          DS_ERR_INVALID_ARG, "caches must be 16-byte aligned");
  REQUIRE(a->workspace, DS_ERR_WORKSPACE, "workspace is NULL");
  REQUIRE(a->workspace_bytes >= ds::kStatusBytes, DS_ERR_WORKSPACE,
          "workspace_bytes %zu < %zu", a->workspace_bytes, ds::kStatusBytes);
  cudaError_t e = ds::launch_compact_append(*a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ds_compact_append launch");
  return ok();
}

}  // extern "C"
