/*
 * ds.h -- C ABI of the GB300 (sm_103a) tree-verify library.
 *
 * The library implements the target-model verify step of long-context
 * speculative decoding with a draft token tree:
 *
 *   ds_verify_attn        split-KV attention of every tree node over a paged
 *                         bf16 KV cache plus causal attention over the node's
 *                         own ancestors, emitting per-chunk attention mass
 *                         ("salience") in the same pass;
 *   ds_chunk_topk_gather  top-k chunks by salience plus a recent window,
 *                         gathered into a compact contiguous cache;
 *   ds_accept             the accepted path: greedy accept-if-equal or exact
 *                         tree rejection sampling with supplied uniforms
 *                         (ds_accept_static: the same over a scratch the
 *                         library owns, for callers that cannot allocate);
 *   ds_kv_commit          the accepted path's tree K/V moved behind the root
 *                         in every layer, and the new context lengths;
 *   ds_compact_append     newly committed tokens appended to the compact
 *                         cache between retrievals.
 *
 * Conventions (all entry points):
 *   - Every pointer named in an args struct is a DEVICE pointer unless its
 *     comment says otherwise.  The caller owns every buffer, including the
 *     workspace; the library never allocates device memory.
 *   - Work is enqueued asynchronously on the caller's stream (`stream` is a
 *     cudaStream_t passed as void*; NULL is the legacy default stream).
 *   - Arguments are validated on the host before any work is enqueued.  A
 *     refused call returns DS_ERR_INVALID_ARG or DS_ERR_UNSUPPORTED and
 *     enqueues nothing; ds_last_error() then names the argument.
 *   - Values that live in device memory (lengths, parents, page ids, tokens)
 *     are checked by the kernels themselves.  A bad value never causes an
 *     out-of-bounds access: the affected sequence is skipped or the access
 *     is replaced by zeros, and a sticky bit is set in the workspace's
 *     status word (see ds_device_status).
 *   - bf16 means IEEE-754 binary32 truncated to its upper 16 bits (round to
 *     nearest even when produced), stored as uint16.
 */
#ifndef DS_VERIFY_H_
#define DS_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DS_ABI_VERSION 2
/* Largest draft tree per sequence: one 64-bit ancestor mask per node. */
#define DS_MAX_TREE_NODES 64

typedef enum {
  DS_OK = 0,
  DS_ERR_INVALID_ARG = 1,  /* a NULL pointer, negative size, bad enum, ...  */
  DS_ERR_UNSUPPORTED = 2,  /* a valid value the library does not support    */
  DS_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed   */
  DS_ERR_TIMEOUT = 4,      /* reserved: a bounded device-side wait gave up  */
  DS_ERR_WORKSPACE = 5     /* workspace missing, misaligned or too small    */
} ds_status;

/* Paged cache layouts.  NHD: [num_pages, page_size, num_kv_heads, head_dim];
 * HND: [num_pages, num_kv_heads, page_size, head_dim].  Both bf16, head_dim
 * contiguous.  Slot t of sequence b lives in page page_table[b][t/page_size]
 * at offset t % page_size. */
typedef enum { DS_KV_NHD = 0, DS_KV_HND = 1 } ds_kv_layout;

typedef enum { DS_OUT_BF16 = 0, DS_OUT_F32 = 1 } ds_out_dtype;

typedef enum { DS_ACCEPT_GREEDY = 0, DS_ACCEPT_REJECT = 1 } ds_accept_mode;

/* Sticky device-side status bits (ds_device_status). */
#define DS_DEV_BAD_LENGTH   0x1u  /* ctx_len < 0, or L+T beyond max_pages*page_size,
                                     or ceil(L/chunk) beyond max_chunks          */
#define DS_DEV_BAD_TREE     0x2u  /* tree size outside [0, 64], offsets not
                                     monotone, or a parent not an earlier node   */
#define DS_DEV_BAD_PAGE     0x4u  /* a page id outside [0, num_pages)            */
#define DS_DEV_BAD_TOKEN    0x8u  /* a draft token outside [0, vocab)            */
#define DS_DEV_TIMEOUT      0x10u /* a bounded wait inside a kernel gave up      */

/* Name of the last failure on the calling thread ("" if none).  The string is
 * owned by the library and valid until the next call on this thread. */
const char* ds_last_error(void);

/* Library ABI version (DS_ABI_VERSION of the build). */
int32_t ds_abi_version(void);

/* sizeof() of each args struct as compiled into the library: 0 verify,
 * 1 gather, 2 accept, 3 commit, 4 append; -1 for anything else.  Bindings compare these with
 * their own struct layouts before the first call. */
int64_t ds_struct_size(int32_t which);

/* Zero the whole workspace: the status word (bytes 0..255 of any workspace)
 * and the verify call's split counters behind it (which every completed
 * call leaves at zero).  Call once after allocating a workspace, whenever the
 * sticky bits should be cleared, and after a call that set DS_DEV_TIMEOUT (an
 * aborted call can leave counters behind).  Enqueued on `stream`. */
ds_status ds_workspace_init(void* workspace, size_t workspace_bytes,
                            void* stream);

/* Copy the workspace's sticky status bits to *flags (host).  Synchronises
 * `stream` first.  0 means every device-side value checked so far was valid. */
ds_status ds_device_status(const void* workspace, uint32_t* flags,
                           void* stream);

/* ------------------------------------------------------------------------ *
 * Tree-verify attention with fused chunk salience.
 *
 * Defines (vllm-diffspec README, "What DiffSpec Does" items 2 and 5 and
 * "Architecture": chunks scored directly from paged target KV without
 * materialising the attention matrix; CGCL-codes/DiffSpec README,
 * "Features": salience-aware chunk encoding; adaptive-specdec README,
 * "Layout": the chain row mask s <= lengths[b] + j):
 *
 *   For sequence b with committed context length L = ctx_lens[b] and tree
 *   nodes n = tree_offsets[b] .. tree_offsets[b+1]-1 (local index j = n -
 *   tree_offsets[b], T = tree size <= 64, parents[n] local, -1 for j = 0),
 *   the tree's own keys and values sit in the paged cache at slots L + j.
 *   Query row (node j, query head h) attends, under kv head h / (Hq/Hkv),
 *   to every context slot t < L and to tree slot L + i iff i is j or an
 *   ancestor of j:
 *       s_t = scale * <q[n, h, :], k_t>,  p = softmax(s),
 *       out[n, h, :] = sum_t p_t v_t.
 *   chunk_scores[b, c] (= or +=, see accumulate_scores) is the attention
 *   mass that context chunk c = [c*C, min((c+1)*C, L)) receives, summed over
 *   all query heads and tree nodes of b, each row normalised by its full
 *   softmax denominator (context plus ancestors).  Only c < ceil(L/C) is
 *   written; other entries of the row are left untouched.
 *
 * Constraints refused with DS_ERR_UNSUPPORTED (by name):
 *   head_dim not 64 or 128; page_size not 16, 32, 64 or 128; chunk_size not
 *   a multiple of page_size or above 128 or not a power of two;
 *   num_q_heads not a multiple of num_kv_heads, or the group size
 *   num_q_heads / num_kv_heads not a power of two up to 16.
 * Alignment: q, caches, out and the workspace 16-byte aligned.
 * ------------------------------------------------------------------------ */
typedef struct ds_verify_args {
  const void*    q;             /* [n_nodes, num_q_heads, head_dim] bf16       */
  const void*    k_cache;       /* paged bf16, layout kv_layout                */
  const void*    v_cache;       /* paged bf16, same layout and page pool       */
  const int32_t* page_table;    /* [batch, max_pages] page ids                 */
  const int32_t* ctx_lens;      /* [batch] committed context length L_b >= 0   */
  const int32_t* tree_offsets;  /* [batch + 1], tree_offsets[0] = 0, last =
                                   n_nodes, nondecreasing                      */
  const int32_t* parents;       /* [n_nodes] local parent, -1 at local 0       */
  int32_t batch;                /* B >= 1                                      */
  int32_t n_nodes;              /* total tree nodes over the batch             */
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;             /* 64 or 128                                   */
  int32_t page_size;
  int32_t num_pages;            /* pages in the pool (bounds page ids)         */
  int32_t max_pages;            /* row length of page_table                    */
  int32_t kv_layout;            /* ds_kv_layout                                */
  int32_t chunk_size;           /* C                                           */
  float   scale;                /* softmax scale; 0 selects 1/sqrt(head_dim)   */
  void*   out;                  /* [n_nodes, num_q_heads, head_dim]            */
  int32_t out_dtype;            /* ds_out_dtype                                */
  float*  chunk_scores;         /* [batch, max_chunks] fp32                    */
  int32_t max_chunks;           /* row length of chunk_scores                  */
  int32_t accumulate_scores;    /* 0: overwrite, 1: add (sum over layers).
                                   With 1 the call is a later layer of the
                                   step that began with 0: ctx_lens and
                                   tree_offsets must hold the same values and
                                   must not be written by the kernel issued
                                   right before this call on `stream` (they
                                   are read while that kernel may still run) */
  int32_t num_sms;              /* CTAs to plan for; 0 = the device's SM count */
  void*   workspace;            /* scratch, >= ds_verify_attn_workspace_size   */
  size_t  workspace_bytes;
  void*   prof_event_start;     /* optional cudaEvent_t (host handle) recorded
                                   on `stream` right before the split-pass
                                   kernel; NULL: not recorded                  */
  void*   prof_event_stop;      /* optional cudaEvent_t recorded right after it */
} ds_verify_args;

/* Fill *args with zeros/NULLs, kv_layout NHD, out_dtype BF16, scale 0. */
void ds_verify_args_default(ds_verify_args* args);

/* Bytes of workspace ds_verify_attn needs for these sizes (host only; reads
 * no pointer).  Depends on batch, n_nodes, head counts, head_dim, page_size,
 * max_pages, chunk_size, max_chunks and num_sms. */
ds_status ds_verify_attn_workspace_size(const ds_verify_args* args,
                                        size_t* bytes);

/* Enqueue the verify step.  Output `out` and `chunk_scores` are complete
 * when the work on `stream` completes.  The workspace must not be shared by
 * calls that may overlap on the GPU.  Its two kernels are launched as
 * programmatic dependents of the preceding work on `stream` (each waits for
 * that work to complete before it reads or writes memory, so ordering is
 * that of the stream; only launch latency overlaps); an event recorded
 * between two calls (for example `prof_event_*`) simply ends that overlap. */
ds_status ds_verify_attn(const ds_verify_args* args, void* stream);

/* ------------------------------------------------------------------------ *
 * Top-k chunk selection plus recent window, gathered into a compact cache.
 *
 * Defines (vllm-diffspec README, "What DiffSpec Does", last paragraph:
 * selected chunks combined with a rolling recent window and rebuilt as a
 * compact cache; CGCL-codes/DiffSpec README, "Features": physically
 * contiguous chunk staging):
 *
 *   ws = max(0, L - window).  Candidates are the chunks wholly before the
 *   window, c with (c+1)*C <= ws.  The min(top_k, #candidates) candidates
 *   with the largest scores[b, c] (ties: lower c) are selected and listed in
 *   ascending order in out_chunk_ids[b, :] (-1 padded).  The working set is
 *   the selected chunks' tokens in ascending order followed by tokens
 *   [ws, L).  Token i of the working set, at absolute position t, is copied
 *   byte for byte from the paged source cache into out_k/out_v[b, i, :, :]
 *   and out_positions[b, i] = t; out_len[b] = working-set size.
 *   out_positions[b, i] = -1 for i >= out_len[b]; out_k/out_v rows beyond
 *   out_len[b] are left untouched.
 *
 *   With rope_base > 0 the source K is pre-RoPE and the compact cache is
 *   rebuilt with local positions (vllm-diffspec README, "Architecture":
 *   dual-view draft cache, canonical pre-RoPE KV at absolute positions and a
 *   compact cache with local draft RoPE positions): row i of out_k is the
 *   source row rotated to position i, pair (j, j + D/2) by the angle
 *   i * rope_base^(-2j/D), j < D/2, rounded to bf16.  The angle is reduced
 *   modulo one turn exactly (64-bit fixed point), its sine and cosine taken
 *   in float32 and the pair rotated in float32, so a value can differ from
 *   the exactly rounded result by one bf16 unit.  V is
 *   always copied byte for byte; rope_base = 0 copies K byte for byte too.
 *
 * Constraints: chunk_size a multiple of page_size; head_dim 64 or 128;
 * capacity >= top_k * chunk_size + window.
 * ------------------------------------------------------------------------ */
typedef struct ds_gather_args {
  const float*   scores;        /* [batch, max_chunks] fp32                    */
  int32_t        max_chunks;
  const int32_t* ctx_lens;      /* [batch]                                     */
  const void*    src_k;         /* paged bf16 source cache (kv_layout)         */
  const void*    src_v;
  const int32_t* page_table;    /* [batch, max_pages]                          */
  int32_t batch;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t num_pages;
  int32_t max_pages;
  int32_t kv_layout;
  int32_t chunk_size;
  int32_t top_k;                /* >= 0                                        */
  int32_t window;               /* >= 0                                        */
  int32_t capacity;             /* rows per sequence in out_k / out_v          */
  void*    out_k;               /* [batch, capacity, num_kv_heads, head_dim]   */
  void*    out_v;
  int32_t* out_positions;       /* [batch, capacity]                           */
  int32_t* out_len;             /* [batch]                                     */
  int32_t* out_chunk_ids;       /* [batch, top_k]                              */
  void*   workspace;            /* scratch, >= ds_chunk_topk_gather_workspace_size */
  size_t  workspace_bytes;
  float   rope_base;            /* 0: no rotation; > 0: RoPE base (theta)      */
} ds_gather_args;

void ds_gather_args_default(ds_gather_args* args);
ds_status ds_chunk_topk_gather_workspace_size(const ds_gather_args* args,
                                              size_t* bytes);
ds_status ds_chunk_topk_gather(const ds_gather_args* args, void* stream);

/* ------------------------------------------------------------------------ *
 * Tree acceptance.
 *
 * Greedy (vllm.cpp docs "Speculative decoding", MTP: accept-if-equal):
 *   from the root (local node 0, whose draft token is ignored) repeatedly
 *   move to the first child, in increasing node index, whose draft token
 *   equals argmax_x target_logits[node, x] (lowest x on ties); stop when no
 *   child does.  bonus = that argmax at the stop node.
 * Rejection (adaptive-specdec README, "Correctness first" and "The
 *   controller"; children of a node are taken to be i.i.d. draws from its
 *   draft distribution):
 *   at node i, p = softmax(target[i]), q = softmax(draft[i]); for each
 *   child c in increasing node index with x = draft_tokens[c]: accept iff
 *   uniforms[c][0] * q(x) < p(x); on rejection p <- max(0, p - q) /
 *   sum(max(0, p - q)) (p kept when that sum is 0).  An accepted child
 *   becomes the current node.  With no child accepted, the bonus token is
 *   the smallest x with sum_{y <= x} p(y) > uniforms[i][1] * sum(p).  A
 *   draft token outside [0, vocab) at a non-root node sets DS_DEV_BAD_TOKEN
 *   and that node is never accepted.
 *
 * Outputs: out_path[b, 0..n-1] = accepted local node ids in order (-1
 * padded to DS_MAX_TREE_NODES), out_n_accepted[b] = n, out_bonus[b].  A
 * sequence with an empty tree gets n = 0 and bonus -1.
 * ------------------------------------------------------------------------ */
typedef struct ds_accept_args {
  int32_t        mode;          /* ds_accept_mode                              */
  const float*   target_logits; /* [n_nodes, vocab] fp32                       */
  const float*   draft_logits;  /* [n_nodes, vocab] fp32; NULL when greedy     */
  const int32_t* draft_tokens;  /* [n_nodes]                                   */
  const int32_t* parents;       /* [n_nodes] local parent, -1 at local 0       */
  const int32_t* tree_offsets;  /* [batch + 1]                                 */
  const float*   uniforms;      /* [n_nodes, 2] in [0, 1); NULL when greedy    */
  int32_t batch;
  int32_t n_nodes;
  int32_t vocab;
  int32_t* out_path;            /* [batch, DS_MAX_TREE_NODES]                  */
  int32_t* out_n_accepted;      /* [batch]                                     */
  int32_t* out_bonus;           /* [batch]                                     */
  void*   workspace;            /* scratch, >= ds_accept_workspace_size        */
  size_t  workspace_bytes;
} ds_accept_args;

void ds_accept_args_default(ds_accept_args* args);
ds_status ds_accept_workspace_size(const ds_accept_args* args, size_t* bytes);
ds_status ds_accept(const ds_accept_args* args, void* stream);

/* Tree acceptance without a caller-supplied workspace.  The method itself
 * has no counterpart to this entry: it is ds_accept for callers that cannot
 * hand out device memory where they call it (a plugin or host callback
 * whose framework owns every allocation and gives it no allocator, or a
 * serving loop that forbids allocation once warm).
 *
 * Same arguments, kernels and results as ds_accept, except that
 * args->workspace must be NULL and args->workspace_bytes 0: the scratch
 * (a status word and one 96-byte record per tree node) is a fixed array in
 * device global memory inside the library, DS_ACCEPT_STATIC_MAX_NODES
 * records long (384 KiB per device).  Nothing is allocated, on the
 * device or through any library, by this call.
 *
 * Refused with DS_ERR_UNSUPPORTED: args->n_nodes > DS_ACCEPT_STATIC_MAX_NODES
 * (use ds_accept).  Refused with DS_ERR_INVALID_ARG: a non-NULL workspace.
 *
 * Every call looks up the array's address in the current context
 * (cudaGetSymbolAddress, which allocates nothing), so a context torn down
 * and created again (cudaDeviceReset) is followed correctly; make one call
 * before capturing `stream` into a graph, so that the module is loaded
 * outside the capture.  Each call then enqueues, on `stream`, a zeroing of
 * the status word (the one part of the scratch that must start at zero;
 * the node records are written before they are read) and the acceptance
 * kernels.
 *
 * flags_out: NULL to return as soon as the work is enqueued; otherwise the
 * call synchronises `stream` and stores this call's device status bits
 * (DS_DEV_BAD_TREE, DS_DEV_BAD_TOKEN; 0 = inputs valid) at *flags_out.
 *
 * One scratch per device: two calls whose work may overlap on the device
 * (different streams, or different host threads, without ordering between
 * them) race on it and give undefined results.  Serialise them. */
#define DS_ACCEPT_STATIC_MAX_NODES 4096
ds_status ds_accept_static(const ds_accept_args* args, uint32_t* flags_out,
                           void* stream);

/* ------------------------------------------------------------------------ *
 * Compact-cache append between retrievals (vllm-diffspec README, "What
 * DiffSpec Does" item 4: KV reuse and locality across decoding steps, and
 * "Configuration": diffspec_retrieval_interval, verifier cycles between
 * retrievals).
 *
 * The compact cache built by ds_chunk_topk_gather is kept; for every
 * sequence b the tokens committed since, t in [from_lens[b], to_lens[b]),
 * are copied from the paged source cache behind its last row: row
 * out_len[b] + (t - from_lens[b]) gets token t, out_positions of that row is
 * t, K is rotated to that row's local position when rope_base > 0 (as in
 * ds_chunk_topk_gather), and out_len[b] grows by to - from.  If the rows do
 * not fit in capacity, or from > to, or to is beyond max_pages * page_size,
 * nothing is appended for b and DS_DEV_BAD_LENGTH is set; a page id outside
 * [0, num_pages) sets DS_DEV_BAD_PAGE and that row is written as zeros.
 * Refused on the host: head_dim not 64 or 128, capacity < 0, rope_base < 0.
 * ------------------------------------------------------------------------ */
typedef struct ds_append_args {
  const void*    src_k;         /* paged bf16 source cache (pre-RoPE K)       */
  const void*    src_v;
  const int32_t* page_table;    /* [batch, max_pages]                         */
  const int32_t* from_lens;     /* [batch]                                    */
  const int32_t* to_lens;       /* [batch]                                    */
  int32_t batch;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t num_pages;
  int32_t max_pages;
  int32_t kv_layout;
  int32_t capacity;             /* rows per sequence of the compact cache     */
  void*    out_k;               /* [batch, capacity, num_kv_heads, head_dim]  */
  void*    out_v;
  int32_t* out_positions;       /* [batch, capacity]                          */
  int32_t* out_len;             /* [batch] rows present; updated in place     */
  float    rope_base;           /* 0: K copied byte for byte                  */
  void*   workspace;            /* >= 256 bytes: the status word              */
  size_t  workspace_bytes;
} ds_append_args;

void ds_append_args_default(ds_append_args* args);
ds_status ds_compact_append(const ds_append_args* args, void* stream);

/* ------------------------------------------------------------------------ *
 * Post-accept KV commit (adaptive-specdec README, "Layout": one cache buffer
 * per layer, a per-sequence lengths vector, writes scattered to each row's
 * own offset, rollback by length).
 *
 * For every sequence b with a tree (T = tree_offsets[b+1] - tree_offsets[b]
 * >= 1) and L = ctx_lens[b]: the root's K/V (node 0) already sits at slot L;
 * the accepted nodes c_1 < ... < c_n (path[b, 0..n-1], n = n_accepted[b], as
 * ds_accept writes them) are copied, in every layer and kv head, K and V,
 * from slot L + c_i to slot L + i, and new_ctx_lens[b] = L + 1 + n.  Slots
 * past the new length keep stale data that the length excludes.  A sequence
 * without a tree gets new_ctx_lens[b] = L.
 *
 * Device-side checks (status bits in the workspace, see ds_device_status):
 * a path that is not strictly increasing inside (0, T) or n outside
 * [0, T-1] sets DS_DEV_BAD_TREE and commits the root only (L + 1); a page id
 * outside [0, num_pages) sets DS_DEV_BAD_PAGE and that slot is skipped;
 * L + T beyond max_pages * page_size sets DS_DEV_BAD_LENGTH and the sequence
 * keeps L.  Refused on the host: num_layers outside 1..DS_MAX_COMMIT_LAYERS,
 * head_dim not 64 or 128, page_size not 16/32/64/128, new_ctx_lens == ctx_lens.
 * Caches as in ds_verify_attn (same layout for all layers), 16-byte aligned.
 * ------------------------------------------------------------------------ */
#define DS_MAX_COMMIT_LAYERS 128

typedef struct ds_commit_args {
  void* const*   k_caches;      /* host array [num_layers] of device pointers   */
  void* const*   v_caches;      /* host array [num_layers] of device pointers   */
  int32_t        num_layers;
  const int32_t* page_table;    /* [batch, max_pages]                           */
  const int32_t* ctx_lens;      /* [batch]                                      */
  const int32_t* tree_offsets;  /* [batch + 1]                                  */
  const int32_t* path;          /* [batch, DS_MAX_TREE_NODES] from ds_accept    */
  const int32_t* n_accepted;    /* [batch]                                      */
  int32_t batch;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t num_pages;
  int32_t max_pages;
  int32_t kv_layout;            /* ds_kv_layout                                 */
  int32_t* new_ctx_lens;        /* [batch] out; must not alias ctx_lens         */
  void*   workspace;            /* >= 256 bytes: the status word                */
  size_t  workspace_bytes;
} ds_commit_args;

void ds_commit_args_default(ds_commit_args* args);
ds_status ds_kv_commit(const ds_commit_args* args, void* stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* DS_VERIFY_H_ */
