"""ds_accept_static: tree acceptance over the library's own static scratch.

The GPU tests call the entry through the C ABI and compare it with
ds_accept (caller workspace) on the same inputs, on two calls in a row, and
pin both against the oracle.  The file name puts it last in collection so
that it also runs after every other GPU test in one process.  The refusals
are host-side checks made before any CUDA call, so they run without a GPU.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from long_context_speculative_ds_gb300 import binding as B
from long_context_speculative_ds_gb300 import synth
from oracle import ref
import helpers as H

DS_ACCEPT_STATIC_MAX_NODES = 4096


def _outputs(st, dev):
    i32 = dict(dtype=torch.int32, device=dev)
    batch = len(st.tree_sizes)
    return (torch.full((batch, B.DS_MAX_TREE_NODES), -7, **i32),
            torch.full((batch,), -7, **i32), torch.full((batch,), -7, **i32))


def _args(mode, inp, outs, workspace=None):
    path, n, bonus = outs
    return B.accept_args(mode, inp.target_logits, inp.draft_tokens, inp.parents,
                         inp.tree_offsets, out_path=path, out_n_accepted=n,
                         out_bonus=bonus, draft_logits=inp.draft_logits,
                         uniforms=inp.uniforms, workspace=workspace)


def _host(outs):
    return [t.cpu().numpy().copy() for t in outs]


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["greedy", "reject"])
def test_static_scratch_matches_workspace_entry(mode):
    wl = synth.tiny_workload(batch=6, vocab=1001, max_depth=8, max_branch=4)
    st, inp, _ = H.build_case(wl, mode=mode, seed=4242, ctx_lens=[32] * 6,
                              tree_sizes=[64, 1, 17, 40, 64, 9], draft="noisy")
    dev = inp.target_logits.device

    # ds_accept with a caller workspace
    outs_ws = _outputs(st, dev)
    a = _args(mode, inp, outs_ws)
    ws = torch.empty(B.ds_accept_workspace_size(a), dtype=torch.uint8, device=dev)
    B.ds_workspace_init(ws)
    a = _args(mode, inp, outs_ws, workspace=ws)
    B.ds_accept(a)
    torch.cuda.synchronize()
    assert B.ds_device_status(ws) == 0
    want = _host(outs_ws)

    lib = B.load()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):           # the second call reuses the same scratch
        outs = _outputs(st, dev)
        s = _args(mode, inp, outs)
        assert s.workspace is None and s.workspace_bytes == 0
        flags = C.c_uint32(0xFFFF)
        rc = lib.ds_accept_static(C.byref(s), C.byref(flags), stream)
        assert rc == B.DS_OK, lib.ds_last_error().decode()
        assert flags.value == 0, call
        got = _host(outs)
        for g, w in zip(got, want):
            np.testing.assert_array_equal(g, w)

    # and both agree with the oracle (greedy bit-exact; rejection away from
    # decisions within 1e-6 of their threshold)
    path, n, bonus = want
    tl = inp.target_logits.cpu().numpy()
    toks = inp.draft_tokens.cpu().numpy()
    g_paths = [list(path[b, :n[b]]) for b in range(len(n))]
    if mode == "greedy":
        rp, rn, rb = ref.greedy_accept(tl, toks, st.parents, st.tree_offsets)
        assert g_paths == rp and list(bonus) == rb
    else:
        rec = []
        rp, rn, rb = ref.rejection_accept(
            tl, inp.draft_logits.cpu().numpy(), toks, st.parents, st.tree_offsets,
            inp.uniforms.cpu().numpy(), record=rec)
        assert H.check_rejection(g_paths, list(bonus), rp, rb, rec, "static") <= 1


@pytest.mark.gpu
def test_static_scratch_reports_bad_token():
    """A draft token outside the vocabulary sets DS_DEV_BAD_TOKEN in this
    call's flags, and the next valid call starts from clean flags again."""
    wl = synth.tiny_workload(batch=2, vocab=256, max_depth=4, max_branch=3)
    st, inp, _ = H.build_case(wl, mode="reject", seed=77, ctx_lens=[32, 32],
                              tree_sizes=[8, 5])
    dev = inp.target_logits.device
    bad = inp.draft_tokens.clone()
    bad[1] = wl.vocab + 3
    lib = B.load()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    for tokens, want in ((bad, B.DS_DEV_BAD_TOKEN), (inp.draft_tokens, 0)):
        path, n, bonus = _outputs(st, dev)
        s = B.accept_args("reject", inp.target_logits, tokens, inp.parents,
                          inp.tree_offsets, out_path=path, out_n_accepted=n,
                          out_bonus=bonus, draft_logits=inp.draft_logits,
                          uniforms=inp.uniforms)
        flags = C.c_uint32(0)
        rc = lib.ds_accept_static(C.byref(s), C.byref(flags), stream)
        assert rc == B.DS_OK, lib.ds_last_error().decode()
        assert flags.value == want


def _host_args(n_nodes):
    a = B.AcceptArgs()
    B.load().ds_accept_args_default(C.byref(a))
    a.batch, a.n_nodes, a.vocab = 1, n_nodes, 8
    return a


def test_static_scratch_refuses_too_many_nodes():
    lib = B.load()
    a = _host_args(DS_ACCEPT_STATIC_MAX_NODES + 1)
    rc = lib.ds_accept_static(C.byref(a), None, None)
    assert rc == B.DS_ERR_UNSUPPORTED
    assert b"DS_ACCEPT_STATIC_MAX_NODES" in lib.ds_last_error()


def test_static_scratch_refuses_a_workspace():
    lib = B.load()
    a = _host_args(4)
    buf = (C.c_uint8 * 512)()
    a.workspace, a.workspace_bytes = C.cast(buf, C.c_void_p), 512
    rc = lib.ds_accept_static(C.byref(a), None, None)
    assert rc == B.DS_ERR_INVALID_ARG
    assert b"workspace must be NULL" in lib.ds_last_error()
