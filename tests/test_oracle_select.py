"""Pins for the oracle's top-k chunk selection and compact gather (CPU only).

Selection is checked against NumPy's stable lexsort (a library routine) on
scores with planted ties; the gather against direct fancy indexing of a dense
view of each sequence's cache.
"""
import numpy as np
import pytest
import torch

from oracle import ref
from long_context_speculative_ds_gb300 import synth
from conftest import bf16_bits


def _lexsort_select(scores, n, k):
    idx = np.arange(n)
    order = np.lexsort((idx, -scores[:n]))   # primary: -score, then index
    return np.sort(order[:min(k, n)])


@pytest.mark.parametrize("seed", range(6))
def test_select_matches_lexsort_with_ties(seed):
    rng = np.random.default_rng(seed)
    C, W, k = 8, 20, 5
    L = int(rng.integers(0, 200))
    n_ch = -(-L // C)
    # coarse values force many exact ties
    scores = rng.integers(0, 4, size=max(n_ch, 1)).astype(np.float64) * 0.25
    n = ref.candidate_count(L, C, W)
    assert n == max(0, (max(0, L - W)) // C)
    got = ref.select_chunks(scores, L, C, k, W)
    np.testing.assert_array_equal(got, _lexsort_select(scores, n, k))


def test_candidate_excludes_chunk_straddling_window():
    # L = 100, W = 30 -> ws = 70; chunk 8 covers [64, 72) and straddles ws.
    assert ref.candidate_count(100, 8, 30) == 8
    pos = ref.working_set_positions([1, 7], 100, 8, 30)
    assert pos == list(range(8, 16)) + list(range(56, 64)) + list(range(70, 100))
    # short context: everything is window, nothing is a candidate
    assert ref.candidate_count(20, 8, 30) == 0
    assert ref.working_set_positions([], 20, 8, 30) == list(range(20))


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_gather_matches_fancy_indexing(layout):
    wl = synth.tiny_workload(batch=3, num_q_heads=4, num_kv_heads=2,
                             head_dim=8, page_size=4, chunk_size=8, top_k=3,
                             window=10, number=71)
    st = synth.make_structure(wl, seed=3, ctx_lens=(61, 9, 33),
                              tree_sizes=(3, 2, 4))
    k, v = synth.make_source_cache(st, layout=layout, seed=4)
    kb, vb = bf16_bits(k), bf16_bits(v)
    rng = np.random.default_rng(1)
    scores = rng.random((3, 8))
    cap = wl.top_k * wl.chunk_size + wl.window
    out = ref.gather_compact(kb, vb, st.page_table.numpy(), st.ctx_lens,
                             scores, wl.page_size, wl.chunk_size, wl.top_k,
                             wl.window, cap, layout=layout)
    for b in range(3):
        L = st.ctx_lens[b]
        # dense [slot, H, D] view of this sequence built by fancy indexing
        pages = st.page_table[b].numpy()
        n_pg = -(-(L + st.tree_sizes[b]) // wl.page_size)
        if layout == "NHD":
            dense_k = kb[pages[:n_pg]].reshape(-1, 2, 8)
        else:
            dense_k = kb[pages[:n_pg]].transpose(0, 2, 1, 3).reshape(-1, 2, 8)
        sel = _lexsort_select(scores[b], ref.candidate_count(L, 8, 10), 3)
        ws = max(0, L - 10)
        pos = np.concatenate([np.arange(c * 8, c * 8 + 8) for c in sel] +
                             [np.arange(ws, L)]).astype(np.int64)
        n = len(pos)
        assert out["out_len"][b] == n
        np.testing.assert_array_equal(out["positions"][b, :n], pos)
        assert (out["positions"][b, n:] == -1).all()
        np.testing.assert_array_equal(out["out_k"][b, :n], dense_k[pos])
        np.testing.assert_array_equal(out["chunk_ids"][b, :len(sel)], sel)
        assert (out["chunk_ids"][b, len(sel):] == -1).all()
