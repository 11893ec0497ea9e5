"""Thin ctypes binding of the C ABI declared in include/ds.h.

Argument marshalling only: tensors become device pointers and sizes, each
call goes straight to the library and a non-zero status raises DSError with
the library's own message.  There is no fallback: without the built library
every entry point raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import torch

from . import build as _build

DS_OK, DS_ERR_INVALID_ARG, DS_ERR_UNSUPPORTED, DS_ERR_CUDA, DS_ERR_TIMEOUT, \
    DS_ERR_WORKSPACE = range(6)
DS_KV_NHD, DS_KV_HND = 0, 1
DS_OUT_BF16, DS_OUT_F32 = 0, 1
DS_ACCEPT_GREEDY, DS_ACCEPT_REJECT = 0, 1
DS_MAX_TREE_NODES = 64
DS_DEV_BAD_LENGTH, DS_DEV_BAD_TREE, DS_DEV_BAD_PAGE, DS_DEV_BAD_TOKEN, \
    DS_DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8, 0x10

_p = C.c_void_p
_i = C.c_int32


class VerifyArgs(C.Structure):
    _fields_ = [("q", _p), ("k_cache", _p), ("v_cache", _p),
                ("page_table", _p), ("ctx_lens", _p), ("tree_offsets", _p),
                ("parents", _p),
                ("batch", _i), ("n_nodes", _i), ("num_q_heads", _i),
                ("num_kv_heads", _i), ("head_dim", _i), ("page_size", _i),
                ("num_pages", _i), ("max_pages", _i), ("kv_layout", _i),
                ("chunk_size", _i), ("scale", C.c_float),
                ("out", _p), ("out_dtype", _i),
                ("chunk_scores", _p), ("max_chunks", _i),
                ("accumulate_scores", _i), ("num_sms", _i),
                ("workspace", _p), ("workspace_bytes", C.c_size_t),
                ("prof_event_start", _p), ("prof_event_stop", _p)]


class GatherArgs(C.Structure):
    _fields_ = [("scores", _p), ("max_chunks", _i), ("ctx_lens", _p),
                ("src_k", _p), ("src_v", _p), ("page_table", _p),
                ("batch", _i), ("num_kv_heads", _i), ("head_dim", _i),
                ("page_size", _i), ("num_pages", _i), ("max_pages", _i),
                ("kv_layout", _i), ("chunk_size", _i), ("top_k", _i),
                ("window", _i), ("capacity", _i),
                ("out_k", _p), ("out_v", _p), ("out_positions", _p),
                ("out_len", _p), ("out_chunk_ids", _p),
                ("workspace", _p), ("workspace_bytes", C.c_size_t),
                ("rope_base", C.c_float)]


class AcceptArgs(C.Structure):
    _fields_ = [("mode", _i), ("target_logits", _p), ("draft_logits", _p),
                ("draft_tokens", _p), ("parents", _p), ("tree_offsets", _p),
                ("uniforms", _p), ("batch", _i), ("n_nodes", _i),
                ("vocab", _i), ("out_path", _p), ("out_n_accepted", _p),
                ("out_bonus", _p), ("workspace", _p),
                ("workspace_bytes", C.c_size_t)]


class CommitArgs(C.Structure):
    _fields_ = [("k_caches", C.POINTER(_p)), ("v_caches", C.POINTER(_p)),
                ("num_layers", _i), ("page_table", _p), ("ctx_lens", _p),
                ("tree_offsets", _p), ("path", _p), ("n_accepted", _p),
                ("batch", _i), ("num_kv_heads", _i), ("head_dim", _i),
                ("page_size", _i), ("num_pages", _i), ("max_pages", _i),
                ("kv_layout", _i), ("new_ctx_lens", _p), ("workspace", _p),
                ("workspace_bytes", C.c_size_t)]


class AppendArgs(C.Structure):
    _fields_ = [("src_k", _p), ("src_v", _p), ("page_table", _p),
                ("from_lens", _p), ("to_lens", _p), ("batch", _i),
                ("num_kv_heads", _i), ("head_dim", _i), ("page_size", _i),
                ("num_pages", _i), ("max_pages", _i), ("kv_layout", _i),
                ("capacity", _i), ("out_k", _p), ("out_v", _p),
                ("out_positions", _p), ("out_len", _p), ("rope_base", C.c_float),
                ("workspace", _p), ("workspace_bytes", C.c_size_t)]


class DSError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"ds status {status}: {message}")
        self.status = status


_LIB: Optional[C.CDLL] = None

EXPORTS = ("ds_last_error", "ds_abi_version", "ds_struct_size",
           "ds_workspace_init", "ds_device_status",
           "ds_verify_args_default", "ds_verify_attn_workspace_size",
           "ds_verify_attn", "ds_gather_args_default",
           "ds_chunk_topk_gather_workspace_size", "ds_chunk_topk_gather",
           "ds_accept_args_default", "ds_accept_workspace_size", "ds_accept",
           "ds_accept_static", "ds_commit_args_default", "ds_kv_commit",
           "ds_append_args_default", "ds_compact_append")


def lib_path() -> str:
    return _build.lib_path()


def load(path: Optional[str] = None) -> C.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or lib_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with "
            "`python -m long_context_speculative_ds_gb300.build`")
    lib = C.CDLL(path)
    lib.ds_last_error.restype = C.c_char_p
    lib.ds_abi_version.restype = C.c_int32
    lib.ds_struct_size.restype = C.c_int64
    lib.ds_struct_size.argtypes = [C.c_int32]
    for name in ("ds_workspace_init", "ds_device_status",
                 "ds_verify_attn_workspace_size", "ds_verify_attn",
                 "ds_chunk_topk_gather_workspace_size", "ds_chunk_topk_gather",
                 "ds_accept_workspace_size", "ds_accept", "ds_accept_static",
                 "ds_kv_commit", "ds_compact_append"):
        getattr(lib, name).restype = C.c_int
    for which, cls in enumerate((VerifyArgs, GatherArgs, AcceptArgs, CommitArgs,
                                 AppendArgs)):
        got = lib.ds_struct_size(which)
        if got != C.sizeof(cls):
            raise RuntimeError(f"struct {cls.__name__}: library has {got} bytes,"
                               f" binding {C.sizeof(cls)}")
    _LIB = lib
    return lib


def _check(status: int):
    if status != DS_OK:
        msg = load().ds_last_error().decode()
        raise DSError(status, msg)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream")
                      else int(stream))


_LAYOUT = {"NHD": DS_KV_NHD, "HND": DS_KV_HND}


def _cache_dims(cache: torch.Tensor, layout: str):
    if layout == "NHD":
        num_pages, page_size, kv_heads, head_dim = cache.shape
    else:
        num_pages, kv_heads, page_size, head_dim = cache.shape
    return num_pages, page_size, kv_heads, head_dim


# ---------------------------------------------------------------------------
def verify_args(q, k_cache, v_cache, page_table, ctx_lens, tree_offsets,
                parents, *, chunk_size: int, out=None, chunk_scores=None,
                workspace=None, kv_layout: str = "NHD", scale: float = 0.0,
                accumulate: bool = False, num_sms: int = 0,
                prof_events=None) -> VerifyArgs:
    a = VerifyArgs()
    load().ds_verify_args_default(C.byref(a))
    num_pages, page_size, kv_heads, head_dim = _cache_dims(k_cache, kv_layout)
    a.q, a.k_cache, a.v_cache = _ptr(q), _ptr(k_cache), _ptr(v_cache)
    a.page_table, a.ctx_lens = _ptr(page_table), _ptr(ctx_lens)
    a.tree_offsets, a.parents = _ptr(tree_offsets), _ptr(parents)
    a.batch = page_table.shape[0]
    a.n_nodes = q.shape[0]
    a.num_q_heads = q.shape[1]
    a.num_kv_heads = kv_heads
    a.head_dim = head_dim
    a.page_size = page_size
    a.num_pages = num_pages
    a.max_pages = page_table.shape[1]
    a.kv_layout = _LAYOUT[kv_layout]
    a.chunk_size = chunk_size
    a.scale = scale
    if out is not None:
        a.out = _ptr(out)
        a.out_dtype = DS_OUT_F32 if out.dtype == torch.float32 else DS_OUT_BF16
    if chunk_scores is not None:
        a.chunk_scores = _ptr(chunk_scores)
        a.max_chunks = chunk_scores.shape[1]
    a.accumulate_scores = 1 if accumulate else 0
    a.num_sms = num_sms
    if workspace is not None:
        a.workspace = _ptr(workspace)
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    if prof_events is not None:
        a.prof_event_start = C.c_void_p(prof_events[0].cuda_event)
        a.prof_event_stop = C.c_void_p(prof_events[1].cuda_event)
    return a


def ds_verify_attn_workspace_size(args: VerifyArgs) -> int:
    n = C.c_size_t(0)
    _check(load().ds_verify_attn_workspace_size(C.byref(args), C.byref(n)))
    return n.value


def ds_verify_attn(args: VerifyArgs, stream=None):
    _check(load().ds_verify_attn(C.byref(args), _stream(stream)))


def gather_args(scores, ctx_lens, src_k, src_v, page_table, *, chunk_size: int,
                top_k: int, window: int, out_k, out_v, out_positions, out_len,
                out_chunk_ids, workspace=None, kv_layout: str = "NHD",
                rope_base: float = 0.0) -> GatherArgs:
    a = GatherArgs()
    load().ds_gather_args_default(C.byref(a))
    num_pages, page_size, kv_heads, head_dim = _cache_dims(src_k, kv_layout)
    a.scores, a.max_chunks = _ptr(scores), scores.shape[1]
    a.ctx_lens = _ptr(ctx_lens)
    a.src_k, a.src_v, a.page_table = _ptr(src_k), _ptr(src_v), _ptr(page_table)
    a.batch = page_table.shape[0]
    a.num_kv_heads, a.head_dim, a.page_size = kv_heads, head_dim, page_size
    a.num_pages, a.max_pages = num_pages, page_table.shape[1]
    a.kv_layout = _LAYOUT[kv_layout]
    a.chunk_size, a.top_k, a.window = chunk_size, top_k, window
    a.capacity = out_k.shape[1]
    a.out_k, a.out_v = _ptr(out_k), _ptr(out_v)
    a.out_positions, a.out_len = _ptr(out_positions), _ptr(out_len)
    a.out_chunk_ids = _ptr(out_chunk_ids)
    a.rope_base = rope_base
    if workspace is not None:
        a.workspace = _ptr(workspace)
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def ds_chunk_topk_gather_workspace_size(args: GatherArgs) -> int:
    n = C.c_size_t(0)
    _check(load().ds_chunk_topk_gather_workspace_size(C.byref(args), C.byref(n)))
    return n.value


def ds_chunk_topk_gather(args: GatherArgs, stream=None):
    _check(load().ds_chunk_topk_gather(C.byref(args), _stream(stream)))


def accept_args(mode: str, target_logits, draft_tokens, parents, tree_offsets,
                *, out_path, out_n_accepted, out_bonus, draft_logits=None,
                uniforms=None, workspace=None) -> AcceptArgs:
    a = AcceptArgs()
    load().ds_accept_args_default(C.byref(a))
    a.mode = DS_ACCEPT_REJECT if mode == "reject" else DS_ACCEPT_GREEDY
    a.target_logits, a.draft_logits = _ptr(target_logits), _ptr(draft_logits)
    a.draft_tokens, a.parents = _ptr(draft_tokens), _ptr(parents)
    a.tree_offsets, a.uniforms = _ptr(tree_offsets), _ptr(uniforms)
    a.batch = tree_offsets.shape[0] - 1
    a.n_nodes = target_logits.shape[0]
    a.vocab = target_logits.shape[1]
    a.out_path, a.out_n_accepted = _ptr(out_path), _ptr(out_n_accepted)
    a.out_bonus = _ptr(out_bonus)
    if workspace is not None:
        a.workspace = _ptr(workspace)
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def ds_accept_workspace_size(args: AcceptArgs) -> int:
    n = C.c_size_t(0)
    _check(load().ds_accept_workspace_size(C.byref(args), C.byref(n)))
    return n.value


def ds_accept(args: AcceptArgs, stream=None):
    _check(load().ds_accept(C.byref(args), _stream(stream)))


def ds_accept_static(args: AcceptArgs, stream=None, read_flags: bool = True):
    """ds_accept over the library's own scratch (args.workspace must be
    unset).  With read_flags the call waits for the stream and returns the
    device status bits of this call; otherwise it returns None at once."""
    flags = C.c_uint32(0)
    _check(load().ds_accept_static(C.byref(args),
                                   C.byref(flags) if read_flags else None,
                                   _stream(stream)))
    return flags.value if read_flags else None


def commit_args(k_caches, v_caches, page_table, ctx_lens, tree_offsets, path,
                n_accepted, *, new_ctx_lens, workspace,
                kv_layout: str = "NHD") -> CommitArgs:
    """Arguments of ds_kv_commit.  k_caches / v_caches are lists of the
    layers' paged caches; the pointer arrays live in the returned struct
    (kept alive by it) and are read on the host at call time."""
    a = CommitArgs()
    load().ds_commit_args_default(C.byref(a))
    nl = len(k_caches)
    kp = (_p * nl)(*[t.data_ptr() for t in k_caches])
    vp = (_p * nl)(*[t.data_ptr() for t in v_caches])
    a._keep = (kp, vp)
    a.k_caches = C.cast(kp, C.POINTER(_p))
    a.v_caches = C.cast(vp, C.POINTER(_p))
    a.num_layers = nl
    num_pages, page_size, kv_heads, head_dim = _cache_dims(k_caches[0], kv_layout)
    a.page_table, a.ctx_lens = _ptr(page_table), _ptr(ctx_lens)
    a.tree_offsets, a.path, a.n_accepted = _ptr(tree_offsets), _ptr(path), _ptr(n_accepted)
    a.batch = page_table.shape[0]
    a.num_kv_heads, a.head_dim, a.page_size = kv_heads, head_dim, page_size
    a.num_pages, a.max_pages = num_pages, page_table.shape[1]
    a.kv_layout = _LAYOUT[kv_layout]
    a.new_ctx_lens = _ptr(new_ctx_lens)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def ds_kv_commit(args: CommitArgs, stream=None):
    _check(load().ds_kv_commit(C.byref(args), _stream(stream)))


def append_args(src_k, src_v, page_table, from_lens, to_lens, *, out_k, out_v,
                out_positions, out_len, workspace, kv_layout: str = "NHD",
                rope_base: float = 0.0) -> AppendArgs:
    a = AppendArgs()
    load().ds_append_args_default(C.byref(a))
    num_pages, page_size, kv_heads, head_dim = _cache_dims(src_k, kv_layout)
    a.src_k, a.src_v, a.page_table = _ptr(src_k), _ptr(src_v), _ptr(page_table)
    a.from_lens, a.to_lens = _ptr(from_lens), _ptr(to_lens)
    a.batch = page_table.shape[0]
    a.num_kv_heads, a.head_dim, a.page_size = kv_heads, head_dim, page_size
    a.num_pages, a.max_pages = num_pages, page_table.shape[1]
    a.kv_layout = _LAYOUT[kv_layout]
    a.capacity = out_k.shape[1]
    a.out_k, a.out_v = _ptr(out_k), _ptr(out_v)
    a.out_positions, a.out_len = _ptr(out_positions), _ptr(out_len)
    a.rope_base = rope_base
    a.workspace = _ptr(workspace)
    a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def ds_compact_append(args: AppendArgs, stream=None):
    _check(load().ds_compact_append(C.byref(args), _stream(stream)))


def ds_workspace_init(workspace: torch.Tensor, stream=None):
    _check(load().ds_workspace_init(_ptr(workspace),
                                    C.c_size_t(workspace.numel()),
                                    _stream(stream)))


def ds_device_status(workspace: torch.Tensor, stream=None) -> int:
    flags = C.c_uint32(0)
    _check(load().ds_device_status(_ptr(workspace), C.byref(flags),
                                   _stream(stream)))
    return flags.value
