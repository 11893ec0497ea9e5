"""Host-side checks of the C ABI (no GPU needed): the library builds, loads,
exports every function include/ds.h declares with matching struct layouts,
and refuses bad arguments by name before touching the device."""
import ctypes as C
import os
import re

import pytest

from long_context_speculative_ds_gb300 import binding as B
from long_context_speculative_ds_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load()


def _declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(ds_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_function(lib):
    declared = _declared_functions()
    assert len(declared) >= 14
    for name in declared:
        assert hasattr(lib, name), name
    assert set(B.EXPORTS) == set(declared)


def test_struct_layouts_and_version(lib):
    assert lib.ds_abi_version() == 2
    assert lib.ds_struct_size(0) == C.sizeof(B.VerifyArgs)
    assert lib.ds_struct_size(1) == C.sizeof(B.GatherArgs)
    assert lib.ds_struct_size(2) == C.sizeof(B.AcceptArgs)
    assert lib.ds_struct_size(3) == C.sizeof(B.CommitArgs)
    assert lib.ds_struct_size(4) == C.sizeof(B.AppendArgs)
    assert lib.ds_struct_size(7) == -1


def _verify_args(**kw):
    a = B.VerifyArgs()
    B.load().ds_verify_args_default(C.byref(a))
    base = dict(batch=1, n_nodes=8, num_q_heads=32, num_kv_heads=8,
                head_dim=128, page_size=16, num_pages=100, max_pages=64,
                chunk_size=64, max_chunks=16, num_sms=152)
    base.update(kw)
    for k, v in base.items():
        setattr(a, k, v)
    return a


def _ws_size(a):
    n = C.c_size_t(0)
    st = B.load().ds_verify_attn_workspace_size(C.byref(a), C.byref(n))
    return st, n.value, B.load().ds_last_error().decode()


@pytest.mark.parametrize("field,value,status,word", [
    ("head_dim", 96, B.DS_ERR_UNSUPPORTED, "head_dim"),
    ("page_size", 24, B.DS_ERR_UNSUPPORTED, "page_size"),
    ("chunk_size", 48, B.DS_ERR_UNSUPPORTED, "chunk_size"),
    ("chunk_size", 8, B.DS_ERR_UNSUPPORTED, "chunk_size"),
    ("chunk_size", 256, B.DS_ERR_UNSUPPORTED, "chunk_size"),
    ("num_q_heads", 36, B.DS_ERR_UNSUPPORTED, "num_q_heads"),
    ("num_q_heads", 24, B.DS_ERR_UNSUPPORTED, "group size"),
    ("batch", 0, B.DS_ERR_INVALID_ARG, "batch"),
    ("kv_layout", 5, B.DS_ERR_INVALID_ARG, "kv_layout"),
    ("out_dtype", 9, B.DS_ERR_INVALID_ARG, "out_dtype"),
    ("num_pages", 0, B.DS_ERR_INVALID_ARG, "num_pages"),
])
def test_verify_refuses_by_name(lib, field, value, status, word):
    st, _, msg = _ws_size(_verify_args(**{field: value}))
    assert st == status and word in msg, (st, msg)
    # the launch entry point refuses identically, before any CUDA call
    st2 = lib.ds_verify_attn(C.byref(_verify_args(**{field: value})), None)
    assert st2 == status


def test_verify_workspace_size_and_null_checks(lib):
    st, n, _ = _ws_size(_verify_args())
    assert st == B.DS_OK and n > 0
    # more chunks or more sequences never shrink the workspace
    assert _ws_size(_verify_args(max_chunks=2048))[1] > n
    assert _ws_size(_verify_args(batch=4))[1] > n
    st = lib.ds_verify_attn(C.byref(_verify_args()), None)
    assert st == B.DS_ERR_INVALID_ARG
    assert "is NULL" in lib.ds_last_error().decode()


def test_gather_and_accept_refusals(lib):
    g = B.GatherArgs()
    lib.ds_gather_args_default(C.byref(g))
    for k, v in dict(batch=1, num_kv_heads=8, head_dim=128, page_size=16,
                     num_pages=10, max_pages=4, chunk_size=64, top_k=4,
                     window=64, capacity=100, max_chunks=8).items():
        setattr(g, k, v)
    n = C.c_size_t(0)
    assert lib.ds_chunk_topk_gather_workspace_size(C.byref(g), C.byref(n)) == \
        B.DS_ERR_INVALID_ARG
    assert "capacity" in lib.ds_last_error().decode()
    g.capacity = 4 * 64 + 64
    assert lib.ds_chunk_topk_gather_workspace_size(C.byref(g), C.byref(n)) == B.DS_OK
    g.rope_base = -1.0
    assert lib.ds_chunk_topk_gather_workspace_size(C.byref(g), C.byref(n)) == \
        B.DS_ERR_INVALID_ARG
    assert "rope_base" in lib.ds_last_error().decode()
    g.rope_base = 0.0
    g.chunk_size = 40
    assert lib.ds_chunk_topk_gather(C.byref(g), None) == B.DS_ERR_UNSUPPORTED

    a = B.AcceptArgs()
    lib.ds_accept_args_default(C.byref(a))
    a.batch, a.n_nodes, a.vocab, a.mode = 1, 4, 100, 7
    assert lib.ds_accept(C.byref(a), None) == B.DS_ERR_INVALID_ARG
    assert "mode" in lib.ds_last_error().decode()
    a.mode = B.DS_ACCEPT_REJECT
    a.target_logits = a.draft_tokens = a.parents = a.tree_offsets = 16
    a.out_path = a.out_n_accepted = a.out_bonus = 16
    assert lib.ds_accept(C.byref(a), None) == B.DS_ERR_INVALID_ARG
    assert "draft_logits" in lib.ds_last_error().decode()
    assert lib.ds_accept_workspace_size(C.byref(a), C.byref(n)) == B.DS_OK
    assert n.value >= 256 + 4 * 48


def _commit_args(**kw):
    a = B.CommitArgs()
    B.load().ds_commit_args_default(C.byref(a))
    ptrs = (C.c_void_p * 2)(256, 512)
    a.k_caches = C.cast(ptrs, C.POINTER(C.c_void_p))
    a.v_caches = C.cast(ptrs, C.POINTER(C.c_void_p))
    base = dict(num_layers=2, batch=1, num_kv_heads=8, head_dim=128, page_size=16,
                num_pages=10, max_pages=4, page_table=16, ctx_lens=32,
                tree_offsets=48, path=64, n_accepted=80, new_ctx_lens=96,
                workspace=4096, workspace_bytes=256)
    base.update(kw)
    for k, v in base.items():
        setattr(a, k, v)
    return a, ptrs


@pytest.mark.parametrize("field,value,status,word", [
    ("num_layers", 0, B.DS_ERR_UNSUPPORTED, "num_layers"),
    ("num_layers", 129, B.DS_ERR_UNSUPPORTED, "num_layers"),
    ("head_dim", 96, B.DS_ERR_UNSUPPORTED, "head_dim"),
    ("page_size", 24, B.DS_ERR_UNSUPPORTED, "page_size"),
    ("batch", 0, B.DS_ERR_INVALID_ARG, "batch"),
    ("kv_layout", 3, B.DS_ERR_INVALID_ARG, "kv_layout"),
    ("new_ctx_lens", 32, B.DS_ERR_INVALID_ARG, "alias"),
    ("path", None, B.DS_ERR_INVALID_ARG, "is NULL"),
    ("workspace_bytes", 8, B.DS_ERR_WORKSPACE, "workspace_bytes"),
])
def test_commit_refuses_by_name(lib, field, value, status, word):
    a, keep = _commit_args(**{field: value})
    st = lib.ds_kv_commit(C.byref(a), None)
    assert st == status and word in lib.ds_last_error().decode(), (st, lib.ds_last_error())


def test_commit_refuses_unaligned_cache(lib):
    a, keep = _commit_args()
    bad = (C.c_void_p * 2)(256, 520)
    a.v_caches = C.cast(bad, C.POINTER(C.c_void_p))
    assert lib.ds_kv_commit(C.byref(a), None) == B.DS_ERR_INVALID_ARG
    assert "16-byte aligned" in lib.ds_last_error().decode()


def _append_args(**kw):
    a = B.AppendArgs()
    B.load().ds_append_args_default(C.byref(a))
    base = dict(src_k=256, src_v=512, page_table=16, from_lens=32, to_lens=48,
                batch=1, num_kv_heads=8, head_dim=128, page_size=16, num_pages=10,
                max_pages=4, capacity=100, out_k=1024, out_v=2048, out_positions=64,
                out_len=80, workspace=4096, workspace_bytes=256)
    base.update(kw)
    for k, v in base.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,status,word", [
    ("head_dim", 32, B.DS_ERR_UNSUPPORTED, "head_dim"),
    ("batch", 0, B.DS_ERR_INVALID_ARG, "batch"),
    ("capacity", -1, B.DS_ERR_INVALID_ARG, "capacity"),
    ("rope_base", -2.0, B.DS_ERR_INVALID_ARG, "rope_base"),
    ("rope_base", float("inf"), B.DS_ERR_INVALID_ARG, "rope_base"),
    ("to_lens", None, B.DS_ERR_INVALID_ARG, "is NULL"),
    ("out_k", 1032, B.DS_ERR_INVALID_ARG, "aligned"),
    ("workspace", None, B.DS_ERR_WORKSPACE, "workspace"),
])
def test_append_refuses_by_name(lib, field, value, status, word):
    st = lib.ds_compact_append(C.byref(_append_args(**{field: value})), None)
    assert st == status and word in lib.ds_last_error().decode(), (st, lib.ds_last_error())
