"""GPU parity of ds_kv_commit, through the C ABI: every layer's paged K and V
bit-exact against the oracle's kv_commit, and the new context lengths.

Cases: random trees with random root-to-node paths (empty, partial, a
sequence whose whole chain is accepted), several layers, both cache
layouts, ragged batches with an empty tree; the path written by ds_accept
on the GPU fed straight into the commit; bad paths and bad page ids flagged
and skipped.
"""
import numpy as np
import pytest
import torch

from long_context_speculative_ds_gb300 import binding as B
from long_context_speculative_ds_gb300 import synth
from oracle import ref
import helpers as H

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _paths(st, rng, chain_full=None):
    """A random root-to-node path per sequence (-1 padded to 64)."""
    out, ns = [], []
    for b in range(len(st.tree_sizes)):
        n0 = st.tree_offsets[b]
        par = [st.parents[n0 + j] for j in range(st.tree_sizes[b])]
        path, i = [], 0
        while par:
            kids = [c for c in range(len(par)) if par[c] == i]
            if not kids or rng.random() < 0.15:
                break
            i = int(kids[rng.integers(0, len(kids))])
            path.append(i)
        out.append(path + [-1] * (64 - len(path)))
        ns.append(len(path))
    return out, ns


def _commit(st, ks, vs, path, ns, layout, ctx_lens=None):
    dev = ks[0].device
    i32 = dict(dtype=torch.int32, device=dev)
    lens = torch.tensor(st.ctx_lens if ctx_lens is None else ctx_lens, **i32)
    new = torch.full_like(lens, -5)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    a = B.commit_args(ks, vs, st.page_table.to(dev), lens,
                      torch.tensor(st.tree_offsets, **i32),
                      torch.tensor(path, **i32), torch.tensor(ns, **i32),
                      new_ctx_lens=new, workspace=ws, kv_layout=layout)
    B.ds_kv_commit(a)
    torch.cuda.synchronize()
    return new.cpu().numpy(), B.ds_device_status(ws)


def _check_layers(st, ks_before, ks_after, vs_before, vs_after, path, ns, layout, new):
    pt = st.page_table.numpy()
    for l in range(len(ks_before)):
        k2, v2, lens = ref.kv_commit(ks_before[l], vs_before[l], pt, st.ctx_lens,
                                     st.tree_offsets, path, ns, st.workload.page_size,
                                     layout)
        assert (k2 == ks_after[l]).all(), f"layer {l} K"
        assert (v2 == vs_after[l]).all(), f"layer {l} V"
        assert list(new) == list(lens)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("seed", [0, 1])
def test_commit_matches_oracle(layout, seed):
    wl = synth.tiny_workload(batch=5, head_dim=128, num_q_heads=8, num_kv_heads=2,
                             max_depth=10, max_branch=3)
    rng = np.random.default_rng(seed)
    trees = [64, 1, 20, 0, 37]
    st = synth.make_structure(wl, seed=50 + seed, ctx_lens=[100, 16, 333, 40, 1000],
                              tree_sizes=trees)
    ks, vs = [], []
    for l in range(3):
        _, k, v = synth.make_layer(st, l, device="cuda", layout=layout, seed=70 + l)
        ks.append(k); vs.append(v)
    path, ns = _paths(st, rng)
    kb = [_bits(k) for k in ks]; vb = [_bits(v) for v in vs]
    new, status = _commit(st, ks, vs, path, ns, layout)
    assert status == 0
    _check_layers(st, kb, [_bits(k) for k in ks], vb, [_bits(v) for v in vs],
                  path, ns, layout, new)


def test_commit_chain_fully_accepted_is_identity():
    wl = synth.tiny_workload(batch=1, head_dim=64)
    T = 9
    st = synth.make_structure(wl, seed=3, ctx_lens=[77], tree_sizes=[T],
                              parents=[-1] + list(range(T - 1)))
    _, k, v = synth.make_layer(st, 0, device="cuda")
    kb, vb = _bits(k), _bits(v)
    path = [list(range(1, T)) + [-1] * (64 - T + 1)]
    new, status = _commit(st, [k], [v], path, [T - 1], "NHD")
    assert status == 0 and list(new) == [77 + T]
    assert (_bits(k) == kb).all() and (_bits(v) == vb).all()


def test_accept_then_commit_pipeline():
    """The path ds_accept writes on the GPU goes straight into ds_kv_commit;
    the oracle does greedy acceptance and the commit on the same inputs."""
    wl = synth.tiny_workload(batch=4, vocab=300, max_depth=8, max_branch=3)
    st, inp, _ = H.build_case(wl, mode="greedy", seed=11, ctx_lens=[64, 200, 33, 500],
                              tree_sizes=[30, 12, 64, 7], draft="noisy", layers=2)
    step = H.make_step(wl, inp, "greedy")
    step.accept()
    torch.cuda.synchronize()
    ks = [k for k in inp.k_cache]; vs = [v for v in inp.v_cache]
    kb = [_bits(k) for k in ks]; vb = [_bits(v) for v in vs]
    dev = ks[0].device
    i32 = dict(dtype=torch.int32, device=dev)
    new = torch.full((4,), -5, **i32)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    a = B.commit_args(ks, vs, inp.page_table, inp.ctx_lens, inp.tree_offsets,
                      step.out_path, step.out_n, new_ctx_lens=new, workspace=ws)
    B.ds_kv_commit(a)
    torch.cuda.synchronize()
    assert B.ds_device_status(ws) == 0
    paths, n, _ = ref.greedy_accept(inp.target_logits.cpu().numpy(),
                                    inp.draft_tokens.cpu().numpy(), st.parents,
                                    st.tree_offsets)
    assert sum(n) > 0
    pad = [p + [-1] * (64 - len(p)) for p in paths]
    _check_layers(st, kb, [_bits(k) for k in ks], vb, [_bits(v) for v in vs],
                  pad, n, "NHD", new.cpu().numpy())


def test_bad_path_commits_root_only():
    wl = synth.tiny_workload(batch=2, head_dim=64)
    st = synth.make_structure(wl, seed=4, ctx_lens=[50, 60], tree_sizes=[6, 6])
    _, k, v = synth.make_layer(st, 0, device="cuda")
    kb, vb = _bits(k), _bits(v)
    path = [[3, 2] + [-1] * 62, [1] + [-1] * 63]
    new, status = _commit(st, [k], [v], path, [2, 7], "NHD")   # decreasing; n > T-1
    assert status & B.DS_DEV_BAD_TREE
    assert list(new) == [51, 61]
    assert (_bits(k) == kb).all() and (_bits(v) == vb).all()


def test_bad_page_flagged():
    wl = synth.tiny_workload(batch=1, head_dim=64)
    st = synth.make_structure(wl, seed=5, ctx_lens=[40], tree_sizes=[10])
    _, k, v = synth.make_layer(st, 0, device="cuda")
    st.page_table[0, 40 // wl.page_size] = st.num_pages + 3    # page of slot L
    path = [[2, 5] + [-1] * 62]
    # only valid if 2 and 5 form a path; the commit does not check parents
    new, status = _commit(st, [k], [v], path, [2], "NHD")
    assert status & B.DS_DEV_BAD_PAGE
    assert list(new) == [43]
