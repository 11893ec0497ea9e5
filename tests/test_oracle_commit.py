"""Pins of the oracle's post-accept KV commit (oracle.ref.kv_commit).

The commit moves the accepted path's tree K/V behind the root and grows the
length by 1 + n (adaptive-specdec README, "Layout": per-row lengths, scatter
writes, rollback by length).  Pinned here against things other than itself:
  * slot contents written out by hand through the page-table definition
    (marker values: tree node j holds the value j + 1);
  * attention equivalence: a query that, before the commit, is a leaf under
    the accepted path (so it sees context + root + path through the tree
    mask) must get the same output as the same query placed, after the
    commit, right behind the new length with no tree (plain context);
  * special cases: a chain with every node accepted moves nothing; n = 0
    commits only the root; no tree keeps the length; a path that is not
    increasing is refused.
"""
import numpy as np
import pytest

from oracle import ref

P = 16


def _layout_cache(pages, H, D, layout, rng, fill=None):
    shape = (pages, P, H, D) if layout == "NHD" else (pages, H, P, D)
    if fill is not None:
        return np.full(shape, fill, dtype=np.uint16)
    return rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)


def _slot(cache, page_row, t, layout):
    pg, off = int(page_row[t // P]), t % P
    return cache[pg, off] if layout == "NHD" else cache[pg, :, off]


def _set_slot(cache, page_row, t, layout, val):
    pg, off = int(page_row[t // P]), t % P
    if layout == "NHD":
        cache[pg, off] = val
    else:
        cache[pg, :, off] = val


def _random_tree(T, rng):
    parents = [-1] + [int(rng.integers(0, j)) for j in range(1, T)]
    return parents


def _root_path(parents, rng, max_len=None):
    """A random root-to-node path: repeatedly step to a random child."""
    path, i = [], 0
    while True:
        kids = [c for c in range(len(parents)) if parents[c] == i]
        if not kids or (max_len is not None and len(path) >= max_len):
            return path
        i = int(kids[rng.integers(0, len(kids))])
        path.append(i)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_marker_slots(layout):
    rng = np.random.default_rng(5)
    H, D = 2, 8
    L, T = 37, 12
    pages = (L + T + P - 1) // P + 3
    page_row = rng.permutation(pages)          # shuffled pool
    k = _layout_cache(pages, H, D, layout, rng)
    v = _layout_cache(pages, H, D, layout, rng)
    for j in range(T):
        _set_slot(k, page_row, L + j, layout, j + 1)
        _set_slot(v, page_row, L + j, layout, 100 + j)
    path = [2, 5, 9, 11]
    pt = np.array([page_row])
    k2, v2, lens = ref.kv_commit(k, v, pt, [L], [0, T],
                                 [path + [-1] * (64 - len(path))], [len(path)], P, layout)
    assert lens.tolist() == [L + 1 + len(path)]
    for t in range(L):                          # context untouched
        assert (_slot(k2, page_row, t, layout) == _slot(k, page_row, t, layout)).all()
    assert (_slot(k2, page_row, L, layout) == 1).all()        # root stays
    for i, c in enumerate(path, start=1):
        assert (_slot(k2, page_row, L + i, layout) == c + 1).all()
        assert (_slot(v2, page_row, L + i, layout) == 100 + c).all()
    for t in range(L + 1 + len(path), L + T):   # stale tail untouched
        assert (_slot(k2, page_row, t, layout) == _slot(k, page_row, t, layout)).all()
    # inputs not modified
    assert (_slot(k, page_row, L + 1, layout) == 2).all()


def test_chain_full_accept_moves_nothing():
    rng = np.random.default_rng(7)
    H, D, L, T = 2, 8, 20, 6
    pages = 4
    page_row = np.arange(pages)
    k = _layout_cache(pages, H, D, "NHD", rng)
    v = _layout_cache(pages, H, D, "NHD", rng)
    path = list(range(1, T))
    k2, v2, lens = ref.kv_commit(k, v, np.array([page_row]), [L], [0, T],
                                 [path + [-1] * (64 - len(path))], [T - 1], P)
    assert (k2 == k).all() and (v2 == v).all()
    assert lens.tolist() == [L + T]


def test_rollback_and_empty_tree():
    rng = np.random.default_rng(8)
    H, D = 1, 8
    pages = 6
    pt = np.array([np.arange(3), np.arange(3, 6)])
    k = _layout_cache(pages, H, D, "NHD", rng)
    v = _layout_cache(pages, H, D, "NHD", rng)
    none = [-1] * 64
    k2, v2, lens = ref.kv_commit(k, v, pt, [10, 30], [0, 4, 4], [none, none], [0, 0], P)
    assert (k2 == k).all() and (v2 == v).all()
    assert lens.tolist() == [11, 30]            # root committed; no tree keeps L


def test_bad_path_refused():
    rng = np.random.default_rng(9)
    k = _layout_cache(4, 1, 8, "NHD", rng)
    for path, n in (([3, 2], 2), ([0], 1), ([6], 1), ([1, 2, 3, 4, 5, 6], 6)):
        with pytest.raises(ValueError):
            ref.kv_commit(k, k, np.array([np.arange(4)]), [10], [0, 6],
                          [path + [-1] * (64 - len(path))], [n], P)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_attention_equivalence(seed):
    """Before: the query is a new leaf under the accepted path, seeing
    context + root + path through the tree mask.  After: the same query sits
    right behind the committed length with no other tree node."""
    rng = np.random.default_rng(seed)
    H_q, H, D = 4, 2, 16
    L, T = 50, 14
    parents = _random_tree(T, rng)
    path = _root_path(parents, rng)
    n = len(path)
    pages = (L + T + 1 + P - 1) // P + 2
    page_row = rng.permutation(pages)
    pt = np.array([page_row])
    # bf16 bit patterns of modest values: random float32 -> bf16 truncation
    def bf16(shape):
        x = rng.standard_normal(shape).astype(np.float32)
        return (x.view(np.uint32) >> 16).astype(np.uint16)
    k = bf16((pages, P, H, D))
    v = bf16((pages, P, H, D))
    q_leaf = bf16((1, H_q, D))
    leaf = T                                  # new node, child of the path's end
    parents_before = parents + [path[-1] if n else 0]
    q_before = np.concatenate([bf16((T, H_q, D)), q_leaf])
    o_before, _, _ = ref.verify_attention(
        ref.bf16_bits_to_f64(q_before), ref.bf16_bits_to_f64(k), ref.bf16_bits_to_f64(v),
        pt, [L], [0, T + 1], parents_before, P, 16)
    # commit the path (the leaf's own K/V row at slot L + T is left alone)
    k2, v2, lens = ref.kv_commit(k, v, pt, [L], [0, T], [path + [-1] * (64 - n)], [n], P)
    L2 = int(lens[0])
    assert L2 == L + 1 + n
    # the query's own K/V must sit at slot L2 after the commit
    _set_slot(k2, page_row, L2, "NHD", _slot(k, page_row, L + T, "NHD"))
    _set_slot(v2, page_row, L2, "NHD", _slot(v, page_row, L + T, "NHD"))
    o_after, _, _ = ref.verify_attention(
        ref.bf16_bits_to_f64(q_leaf), ref.bf16_bits_to_f64(k2), ref.bf16_bits_to_f64(v2),
        pt, [L2], [0, 1], [-1], P, 16)
    np.testing.assert_allclose(o_after[0], o_before[T], rtol=1e-12, atol=1e-14)
