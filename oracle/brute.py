"""Brute-force checks for the oracle, in pure-Python loops (tiny inputs only).

TEST INFRASTRUCTURE ONLY: used by the tests to pin oracle.ref, never by the
product path.

dense_tree_attention builds the full dense visibility mask over every cache
slot of a sequence, rows x (L + T), from the parent array by following parent
links one at a time, and evaluates softmax attention and chunk masses with
math.exp and explicit sums.  It shares no code with oracle.ref.

greedy_by_paths enumerates every root-to-leaf path of the tree and returns
the longest prefix of one on which every node's token equals the argmax of
its parent's target logits.  With pairwise-distinct sibling tokens exactly one
child can match at each node, so this is the unique greedy-accepted path.
"""
from __future__ import annotations

import math
from typing import List, Sequence


def _is_ancestor_or_self(parents: Sequence[int], i: int, j: int) -> bool:
    """Walk parent links from j up to the root looking for i."""
    n = j
    while n != -1:
        if n == i:
            return True
        n = int(parents[n])
    return False


def dense_tree_attention(q, K, V, L: int, parents: Sequence[int],
                         scale: float, chunk_size: int):
    """One sequence, one query head: q [T][D], K, V [L+T][D] (lists of
    floats) already resolved through the page table.  Returns (o [T][D],
    chunk_mass [ceil(L/C)], tree_mass)."""
    T = len(q)
    D = len(q[0]) if T else 0
    n_slots = L + T
    mask = [[False] * n_slots for _ in range(T)]
    for j in range(T):
        for t in range(n_slots):
            if t < L:
                mask[j][t] = True
            else:
                mask[j][t] = _is_ancestor_or_self(parents, t - L, j)
    n_ch = -(-L // chunk_size)
    chunk_mass = [0.0] * n_ch
    tree_mass = 0.0
    out = []
    for j in range(T):
        logits = []
        for t in range(n_slots):
            if mask[j][t]:
                s = 0.0
                for d in range(D):
                    s += q[j][d] * K[t][d]
                logits.append(s * scale)
            else:
                logits.append(None)
        m = max(x for x in logits if x is not None)
        w = [0.0 if x is None else math.exp(x - m) for x in logits]
        z = sum(w)
        p = [x / z for x in w]
        row = [0.0] * D
        for t in range(n_slots):
            for d in range(D):
                row[d] += p[t] * V[t][d]
        out.append(row)
        for t in range(L):
            chunk_mass[t // chunk_size] += p[t]
        for t in range(L, n_slots):
            tree_mass += p[t]
    return out, chunk_mass, tree_mass


def _argmax(xs) -> int:
    best = 0
    for i in range(1, len(xs)):
        if xs[i] > xs[best]:
            best = i
    return best


def greedy_by_paths(target_logits, draft_tokens, parents: Sequence[int]):
    """Returns (path, bonus) for one tree: local node ids."""
    T = len(parents)
    kids = {i: [] for i in range(T)}
    for c in range(1, T):
        kids[int(parents[c])].append(c)
    leaves_paths: List[List[int]] = []

    def walk(n, acc):
        if not kids[n]:
            leaves_paths.append(acc)
        for c in kids[n]:
            walk(c, acc + [c])

    walk(0, [])
    best: List[int] = []
    for path in leaves_paths:
        prev = 0
        good = []
        for c in path:
            if int(draft_tokens[c]) == _argmax(list(target_logits[prev])):
                good.append(c)
                prev = c
            else:
                break
        if len(good) > len(best):
            best = good
    stop = best[-1] if best else 0
    return best, _argmax(list(target_logits[stop]))
