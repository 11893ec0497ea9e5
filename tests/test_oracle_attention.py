"""Pins for the oracle's verify attention and chunk scores (CPU only).

Each check reaches the oracle's answer another way: pure-Python dense-mask
brute force, the chain special case against a library attention call with the
row mask s <= L + j (adaptive-specdec README, "Layout"), plain decode for a
single node, page-table permutation invariance, closed forms for K = 0 and
V = const, and the total-mass invariant of the chunk scores.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import brute, ref
from long_context_speculative_ds_gb300 import synth
from conftest import bf16_to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small(seed, B=2, Hq=4, Hkv=2, D=8, P=4, ctx=(13, 0), trees=(5, 3),
           C=4, layout="NHD", depth=3, branch=3):
    wl = synth.tiny_workload(batch=B, num_q_heads=Hq, num_kv_heads=Hkv,
                             head_dim=D, page_size=P, chunk_size=C,
                             max_depth=depth, max_branch=branch,
                             window=4, top_k=2, number=70 + seed)
    st = synth.make_structure(wl, seed=seed, ctx_lens=ctx, tree_sizes=trees)
    q, k, v = synth.make_layer(st, 0, layout=layout, seed=seed + 5, plant=False)
    return wl, st, bf16_to_f64(q), bf16_to_f64(k), bf16_to_f64(v)


def _run_ref(wl, st, q, k, v, layout="NHD", scale=None):
    return ref.verify_attention(q, k, v, st.page_table.numpy(), st.ctx_lens,
                                st.tree_offsets, st.parents, wl.page_size,
                                wl.chunk_size, scale=scale, layout=layout)


@pytest.mark.parametrize("seed,ctx,trees,layout", [
    (1, (13, 0), (5, 3), "NHD"),
    (2, (16, 7), (1, 6), "HND"),
    (3, (9, 21), (6, 2), "NHD"),
    (4, (0, 0), (3, 1), "HND"),
])
def test_attention_matches_dense_brute_force(seed, ctx, trees, layout):
    wl, st, q, k, v = _small(seed, ctx=ctx, trees=trees, layout=layout)
    o, scores, tmass = _run_ref(wl, st, q, k, v, layout)
    G = wl.num_q_heads // wl.num_kv_heads
    scale = 1.0 / math.sqrt(wl.head_dim)
    for b in range(wl.batch):
        L = st.ctx_lens[b]
        n0, n1 = st.tree_offsets[b], st.tree_offsets[b + 1]
        K = ref.paged_rows(k, st.page_table[b].numpy(), L + n1 - n0,
                           wl.page_size, layout)
        V = ref.paged_rows(v, st.page_table[b].numpy(), L + n1 - n0,
                           wl.page_size, layout)
        par = st.parents[n0:n1]
        ch_tot = np.zeros(-(-L // wl.chunk_size))
        tm = 0.0
        for h in range(wl.num_q_heads):
            ob, cm, t = brute.dense_tree_attention(
                q[n0:n1, h].tolist(), K[:, h // G].tolist(),
                V[:, h // G].tolist(), L, par, scale, wl.chunk_size)
            np.testing.assert_allclose(o[n0:n1, h], np.array(ob), rtol=1e-12,
                                       atol=1e-12)
            ch_tot += np.array(cm)
            tm += t
        np.testing.assert_allclose(scores[b, :len(ch_tot)], ch_tot, rtol=1e-12,
                                   atol=1e-13)
        assert abs(tmass[b] - tm) < 1e-12


def test_chain_tree_is_causal_decode():
    """parents[j] = j - 1 turns the tree into T ordinary decode tokens: row j
    sees slots s <= L + j.  Checked against torch's SDPA in float64."""
    T, L = 6, 19
    wl, st, q, k, v = _small(7, B=1, ctx=(L,), trees=(T,))
    st.parents = [-1] + list(range(T - 1))
    o, _, _ = _run_ref(wl, st, q, k, v)
    G = wl.num_q_heads // wl.num_kv_heads
    K = ref.paged_rows(k, st.page_table[0].numpy(), L + T, wl.page_size, "NHD")
    V = ref.paged_rows(v, st.page_table[0].numpy(), L + T, wl.page_size, "NHD")
    s = torch.arange(L + T)[None, :]
    j = torch.arange(T)[:, None]
    mask = s <= L + j
    for h in range(wl.num_q_heads):
        qq = torch.from_numpy(q[:, h])[None, None]
        kk = torch.from_numpy(K[:, h // G])[None, None]
        vv = torch.from_numpy(V[:, h // G])[None, None]
        lib = torch.nn.functional.scaled_dot_product_attention(
            qq, kk, vv, attn_mask=mask)[0, 0].numpy()
        np.testing.assert_allclose(o[:, h], lib, rtol=1e-12, atol=1e-12)


def test_single_node_is_plain_decode():
    L = 23
    wl, st, q, k, v = _small(8, B=1, ctx=(L,), trees=(1,))
    o, _, _ = _run_ref(wl, st, q, k, v)
    G = wl.num_q_heads // wl.num_kv_heads
    K = ref.paged_rows(k, st.page_table[0].numpy(), L + 1, wl.page_size, "NHD")
    V = ref.paged_rows(v, st.page_table[0].numpy(), L + 1, wl.page_size, "NHD")
    for h in range(wl.num_q_heads):
        lib = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[:, h])[None, None],
            torch.from_numpy(K[:, h // G])[None, None],
            torch.from_numpy(V[:, h // G])[None, None])[0, 0].numpy()
        np.testing.assert_allclose(o[:, h], lib, rtol=1e-12, atol=1e-12)


def test_page_permutation_invariance():
    wl, st, q, k, v = _small(9, B=2, ctx=(17, 9), trees=(4, 5))
    o1, s1, _ = _run_ref(wl, st, q, k, v)
    # Move every page to a new physical slot and rewrite the table to match.
    rng = np.random.default_rng(0)
    perm = rng.permutation(k.shape[0])
    k2 = np.empty_like(k); v2 = np.empty_like(v)
    k2[perm] = k; v2[perm] = v
    table = st.page_table.numpy().copy()
    valid = table >= 0
    table[valid] = perm[table[valid]]
    o2, s2, _ = ref.verify_attention(q, k2, v2, table, st.ctx_lens,
                                     st.tree_offsets, st.parents,
                                     wl.page_size, wl.chunk_size)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2)


def test_zero_keys_give_mean_of_visible_values_and_closed_form_scores():
    """K = 0 makes every visible key equally likely: o is the mean of the
    visible V rows, and row (j, h) puts 1/(L + depth_j + 1) on each context
    key."""
    wl, st, q, k, v = _small(10, B=2, ctx=(14, 5), trees=(5, 4))
    k = np.zeros_like(k)
    o, scores, tmass = _run_ref(wl, st, q, k, v)
    G = wl.num_q_heads // wl.num_kv_heads
    C = wl.chunk_size
    for b in range(wl.batch):
        L = st.ctx_lens[b]
        n0, n1 = st.tree_offsets[b], st.tree_offsets[b + 1]
        T = n1 - n0
        V = ref.paged_rows(v, st.page_table[b].numpy(), L + T, wl.page_size,
                           "NHD")
        depth = ref.node_depths(st.parents[n0:n1])
        expect_scores = np.zeros(-(-L // C))
        for j in range(T):
            # visible tree slots: walk up to the root
            vis = list(range(L))
            n = j
            while n != -1:
                vis.append(L + n)
                n = st.parents[n0 + n]
            assert len(vis) == L + depth[j] + 1
            for h in range(wl.num_q_heads):
                np.testing.assert_allclose(o[n0 + j, h],
                                           V[vis, h // G].mean(axis=0),
                                           rtol=1e-12, atol=1e-13)
            for c in range(len(expect_scores)):
                size = min((c + 1) * C, L) - c * C
                expect_scores[c] += wl.num_q_heads * size / (L + depth[j] + 1)
        np.testing.assert_allclose(scores[b, :len(expect_scores)],
                                   expect_scores, rtol=1e-12)


def test_constant_values_give_constant_output():
    wl, st, q, k, v = _small(11, B=1, ctx=(11,), trees=(6,))
    v = np.full_like(v, 0.375)
    o, _, _ = _run_ref(wl, st, q, k, v)
    np.testing.assert_allclose(o, 0.375, rtol=1e-13)


@pytest.mark.parametrize("seed", [12, 13])
def test_chunk_mass_plus_tree_mass_is_rows(seed):
    """Every row's softmax sums to one: sum_c score_c + tree mass = T * H_q."""
    wl, st, q, k, v = _small(seed, B=2, ctx=(30, 7), trees=(6, 3))
    _, scores, tmass = _run_ref(wl, st, q, k, v)
    for b in range(wl.batch):
        T = st.tree_sizes[b]
        assert abs(scores[b].sum() + tmass[b] - T * wl.num_q_heads) < 1e-10


def test_golden_worked_attention():
    """Hand-derived worked example (fixture cites its source)."""
    with open(os.path.join(GOLDEN, "attention_worked.json")) as f:
        g = json.load(f)
    q = np.array(g["q"], dtype=np.float64)          # [T, H_q=1, D]
    k = np.array(g["k_cache"], dtype=np.float64)    # [pages, P, 1, D]
    v = np.array(g["v_cache"], dtype=np.float64)
    o, scores, tmass = ref.verify_attention(
        q, k, v, np.array(g["page_table"]), g["ctx_lens"], g["tree_offsets"],
        g["parents"], g["page_size"], g["chunk_size"], scale=g["scale"])
    np.testing.assert_allclose(o, np.array(g["expect_o"]), rtol=1e-12)
    np.testing.assert_allclose(scores, np.array(g["expect_scores"]), rtol=1e-12)
    np.testing.assert_allclose(tmass, np.array(g["expect_tree_mass"]),
                               rtol=1e-12)
