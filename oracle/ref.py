"""Float64 CPU oracle for the target-model tree-verify step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes this module; only the tests, the smoke check and the benchmark's
CPU-baseline leg do.  It shares no code with the CUDA library.

Everything here is the plain definition written out in NumPy float64, step by
step, with no blocking, fusion or reordering:

  * verify_attention: every query row (tree node j, query head h) attends over
    its sequence's committed context positions 0..L-1 (found through the page
    table) and over the tree keys of its ancestors and itself, which sit in the
    same paged cache at slots L..L+T-1 in node order.  Softmax with scale
    1/sqrt(D) unless given.  (vllm-diffspec README, "What DiffSpec Does" items
    2 and 5, and "Architecture": "scores ... chunks from paged target KV
    without materializing the full attention matrix"; the chain special case is
    the row mask s <= lengths[b] + j of adaptive-specdec README, "Layout".)
  * chunk scores: the attention mass each fixed-size context chunk receives,
    summed over query heads and tree nodes, normalised by each row's full
    softmax denominator (context plus ancestors).  Tree keys belong to no chunk.
    (CGCL-codes/DiffSpec README, "Features": salience-aware chunk encoding;
    vllm-diffspec README, "Architecture": target-guided retrieval.)
  * select_chunks / gather_compact: top-k chunks strictly before the recent
    window plus the window itself, copied byte for byte into a compact
    contiguous cache in position order (vllm-diffspec README, "What DiffSpec
    Does", last paragraph: "combined with a rolling recent window, and rebuilt
    as a compact ... cache"; CGCL-codes/DiffSpec README, "Features": chunk
    arena, "physically contiguous chunk staging").
  * rope_rotate / f64_to_bf16_bits: with a RoPE base the gathered pre-RoPE
    K is rotated to its local position in the compact cache (half-split
    pairing, inverse frequencies base^(-2j/D)) and rounded once to bf16.
  * greedy_accept: accept-if-equal against the target argmax, walking the tree
    from the root (vllm.cpp docs "Speculative decoding", section "MTP":
    "greedy decoding plus accept-if-equal rejection").
  * compact_append: between retrievals the tokens committed since are
    appended behind the compact cache's last row (vllm-diffspec README,
    "What DiffSpec Does" item 4; "Configuration", retrieval interval).
  * kv_commit: after acceptance the accepted path's tree K/V move into the
    consecutive slots after the root and the length grows by 1 + n; the
    stale tail is excluded by the length (adaptive-specdec README, "Layout").
  * rejection_accept: accept x ~ q with probability min(1, p(x)/q(x)); on
    rejection continue from the residual norm(max(0, p - q)) (adaptive-specdec
    README, "Correctness first" and "The controller"; Leviathan et al. 2023),
    extended to sibling candidates that were drawn i.i.d. from q.

Readings taken where the pages are silent (listed in the design notes too):
scale 1/sqrt(D); tree K/V in the paged cache at slots L..L+T-1; node 0 is the
root (last committed token) and is a query row but is never itself verified;
the partial last context chunk keeps its own index; a chunk that straddles the
window start is not a candidate; top-k ties go to the lower chunk index; argmax
ties go to the lower token id; duplicate sibling tokens go to the lower node
index; accept iff u*q(x) < p(x) (strict); the bonus token is the smallest x
with cumsum(p)[x] > u * sum(p); a zero residual keeps p unchanged.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np


# --------------------------------------------------------------------------
# helpers

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact upcast of raw bf16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def ancestor_matrix(parents_local: Sequence[int]) -> np.ndarray:
    """anc[j, i] is True iff node i is node j or one of its ancestors.

    parents_local[0] must be -1 (the root) and 0 <= parents_local[j] < j for
    j > 0 (topological order, as the draft-tree parent array is given)."""
    T = len(parents_local)
    anc = np.zeros((T, T), dtype=bool)
    for j in range(T):
        p = int(parents_local[j])
        if j == 0:
            if p != -1:
                raise ValueError("node 0 must be the root (parent -1)")
        elif not (0 <= p < j):
            raise ValueError(f"parent[{j}]={p} is not an earlier node")
        anc[j, j] = True
        if p >= 0:
            anc[j] |= anc[p]
    return anc


def node_depths(parents_local: Sequence[int]) -> List[int]:
    d = []
    for j, p in enumerate(parents_local):
        d.append(0 if p < 0 else d[p] + 1)
    return d


def paged_rows(cache: np.ndarray, page_row: np.ndarray, n_slots: int,
               page_size: int, layout: str) -> np.ndarray:
    """Rows [n_slots, H_kv, D] of one sequence, slot t at page_row[t // P],
    offset t % P.  NHD cache: [pages, P, H_kv, D]; HND: [pages, H_kv, P, D]."""
    t = np.arange(n_slots)
    page = np.asarray(page_row, dtype=np.int64)[t // page_size]
    off = t % page_size
    if layout == "NHD":
        return cache[page, off]
    if layout == "HND":
        return cache[page, :, off]
    raise ValueError(layout)


# --------------------------------------------------------------------------
# verify attention + chunk scores

def verify_attention(q, k_cache, v_cache, page_table, ctx_lens, tree_offsets,
                     parents, page_size: int, chunk_size: int,
                     scale: Optional[float] = None, layout: str = "NHD",
                     max_chunks: Optional[int] = None):
    """Returns (o [n_nodes, H_q, D], scores [B, max_chunks], tree_mass [B]).

    q: [n_nodes, H_q, D]; k_cache, v_cache: paged caches (float64 values of the
    bf16 inputs); page_table [B, max_pages]; ctx_lens [B]; tree_offsets [B+1];
    parents [n_nodes] (local indices).  tree_mass[b] is the total attention
    mass that sequence b's rows put on tree keys (used by the mass invariant).
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    n_nodes, H_q, D = q.shape
    H_kv = k_cache.shape[2] if layout == "NHD" else k_cache.shape[1]
    G = H_q // H_kv
    B = len(ctx_lens)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    n_ch = [-(-int(L) // chunk_size) for L in ctx_lens]
    if max_chunks is None:
        max_chunks = max(n_ch) if n_ch else 0
    o = np.zeros((n_nodes, H_q, D))
    scores = np.zeros((B, max_chunks))
    tree_mass = np.zeros(B)
    for b in range(B):
        L = int(ctx_lens[b])
        n0, n1 = int(tree_offsets[b]), int(tree_offsets[b + 1])
        T = n1 - n0
        if T == 0:
            continue
        anc = ancestor_matrix(parents[n0:n1])
        K = paged_rows(k_cache, page_table[b], L + T, page_size, layout)
        V = paged_rows(v_cache, page_table[b], L + T, page_size, layout)
        # visible[j, t]: context keys are seen by every node, tree key L+i by
        # node j iff i is j or an ancestor of j.
        visible = np.ones((T, L + T), dtype=bool)
        visible[:, L:] = anc
        for h in range(H_q):
            hk = h // G
            s = (q[n0:n1, h, :] @ K[:, hk, :].T) * scale          # [T, L+T]
            s = np.where(visible, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            e = np.exp(s)
            p = e / e.sum(axis=1, keepdims=True)
            o[n0:n1, h, :] = p @ V[:, hk, :]
            for c in range(n_ch[b]):
                scores[b, c] += p[:, c * chunk_size:min((c + 1) * chunk_size, L)].sum()
            tree_mass[b] += p[:, L:].sum()
    return o, scores, tree_mass


# --------------------------------------------------------------------------
# top-k chunk selection + compact gather

def candidate_count(L: int, chunk_size: int, window: int) -> int:
    """Chunks c with (c+1)*C <= ws, ws = max(0, L - W): wholly before the
    recent window."""
    ws = max(0, L - window)
    return ws // chunk_size


def select_chunks(scores_row, L: int, chunk_size: int, top_k: int,
                  window: int) -> List[int]:
    """Top-k candidate chunks by score (ties: lower index), returned in
    ascending chunk order."""
    n = candidate_count(L, chunk_size, window)
    order = sorted(range(n), key=lambda c: (-float(scores_row[c]), c))
    return sorted(order[:min(top_k, n)])


def working_set_positions(chunks: Sequence[int], L: int, chunk_size: int,
                          window: int) -> List[int]:
    """Absolute token positions of the working set, in position order: the
    selected chunks' tokens, then the window [ws, L)."""
    ws = max(0, L - window)
    pos = []
    for c in chunks:
        pos.extend(range(c * chunk_size, (c + 1) * chunk_size))
    pos.extend(range(ws, L))
    return pos


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even), in one step
    (no intermediate float32 rounding); returns uint16 bit patterns.  Finite
    normal-range inputs only."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                 # x = m * 2^e, 0.5 <= |m| < 1
    q = np.rint(m * 256.0)             # 8 significant bits, ties to even
    r = np.ldexp(q / 256.0, e)         # exactly representable in bf16
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def rope_rotate(x, pos: int, base: float) -> np.ndarray:
    """Rotary position embedding of the rows x[..., D] at position `pos`, in
    float64: pair (j, j + D/2) is rotated by the angle pos * base^(-2j/D),
    j < D/2 (the half-split pairing).  Returns float64 (no rounding)."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    j = np.arange(D // 2, dtype=np.float64)
    ang = pos * base ** (-2.0 * j / D)
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :D // 2], x[..., D // 2:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def gather_compact(src_k_bits, src_v_bits, page_table, ctx_lens, scores,
                   page_size: int, chunk_size: int, top_k: int, window: int,
                   capacity: int, layout: str = "NHD", rope_base: float = 0.0):
    """Returns dict with chunk_ids [B, top_k] (-1 padded), positions [B, cap]
    (-1 padded), out_len [B], out_k/out_v [B, cap, H_kv, D] uint16 bits (zero
    beyond out_len).

    With rope_base > 0 the source K is taken to be pre-RoPE and compact row i
    gets RoPE at its local position i (rounded once to bf16): the compact
    cache is rebuilt with local draft positions (vllm-diffspec README,
    "Architecture", dual-view draft cache; "What DiffSpec Does", last
    paragraph).  V is copied unchanged."""
    src_k_bits = np.asarray(src_k_bits)
    src_v_bits = np.asarray(src_v_bits)
    B = len(ctx_lens)
    H_kv = src_k_bits.shape[2] if layout == "NHD" else src_k_bits.shape[1]
    D = src_k_bits.shape[3]
    chunk_ids = np.full((B, top_k), -1, dtype=np.int32)
    positions = np.full((B, capacity), -1, dtype=np.int32)
    out_len = np.zeros(B, dtype=np.int32)
    out_k = np.zeros((B, capacity, H_kv, D), dtype=np.uint16)
    out_v = np.zeros((B, capacity, H_kv, D), dtype=np.uint16)
    for b in range(B):
        L = int(ctx_lens[b])
        sel = select_chunks(scores[b], L, chunk_size, top_k, window)
        chunk_ids[b, :len(sel)] = sel
        pos = working_set_positions(sel, L, chunk_size, window)
        if len(pos) > capacity:
            raise ValueError("capacity too small")
        out_len[b] = len(pos)
        for i, t in enumerate(pos):
            page = int(page_table[b][t // page_size])
            off = t % page_size
            positions[b, i] = t
            if layout == "NHD":
                out_k[b, i] = src_k_bits[page, off]
                out_v[b, i] = src_v_bits[page, off]
            else:
                out_k[b, i] = src_k_bits[page, :, off]
                out_v[b, i] = src_v_bits[page, :, off]
            if rope_base > 0:
                out_k[b, i] = f64_to_bf16_bits(
                    rope_rotate(bf16_bits_to_f64(out_k[b, i]), i, rope_base))
    return dict(chunk_ids=chunk_ids, positions=positions, out_len=out_len,
                out_k=out_k, out_v=out_v)


def compact_append(compact: Dict, src_k_bits, src_v_bits, page_table, from_lens,
                   to_lens, page_size: int, layout: str = "NHD",
                   rope_base: float = 0.0) -> Dict:
    """Between retrievals the compact cache is kept and the tokens committed
    since, [from_lens[b], to_lens[b]), are appended behind its last row, K
    rotated to the appended rows' local positions (vllm-diffspec README,
    "What DiffSpec Does" item 4, KV reuse across decoding steps; the
    retrieval interval of "Configuration").  Returns a new dict; a sequence
    whose rows would not fit is left unchanged (the caller retrieves anew)."""
    out = {k: np.array(v, copy=True) for k, v in compact.items()}
    cap = out["positions"].shape[1]
    for b in range(len(from_lens)):
        f, t = int(from_lens[b]), int(to_lens[b])
        n0 = int(out["out_len"][b])
        if f < 0 or t < f or n0 + (t - f) > cap:
            continue
        for k, pos in enumerate(range(f, t)):
            i = n0 + k
            page = int(page_table[b][pos // page_size])
            off = pos % page_size
            if layout == "NHD":
                rk, rv = src_k_bits[page, off], src_v_bits[page, off]
            else:
                rk, rv = src_k_bits[page, :, off], src_v_bits[page, :, off]
            out["out_k"][b, i] = rk
            out["out_v"][b, i] = rv
            if rope_base > 0:
                out["out_k"][b, i] = f64_to_bf16_bits(
                    rope_rotate(bf16_bits_to_f64(rk), i, rope_base))
            out["positions"][b, i] = pos
        out["out_len"][b] = n0 + (t - f)
    return out


# --------------------------------------------------------------------------
# post-accept KV commit

def kv_commit(k_bits, v_bits, page_table, ctx_lens, tree_offsets, path,
              n_accepted, page_size: int, layout: str = "NHD"):
    """Commit the accepted path of every sequence into its context, for one
    layer's paged cache (raw bf16 bit patterns, any integer dtype).

    The tree's K/V sit at slots L..L+T-1 in node order (node 0, the root, is
    the last committed token and already sits at slot L).  The accepted nodes
    c_1 < ... < c_n (path[b, :n]) move to the consecutive slots L+1..L+n and
    the context length becomes L + 1 + n; the stale slots beyond it are simply
    excluded by the length (adaptive-specdec README, "Layout": one buffer per
    layer, a per-row lengths vector, writes scattered to each row's own
    offset, rollback by length).  Sequences without a tree keep L.

    Returns (k_out, v_out, new_lens) with the inputs left untouched."""
    k_out = np.array(k_bits, copy=True)
    v_out = np.array(v_bits, copy=True)
    B = len(ctx_lens)
    new_lens = np.zeros(B, dtype=np.int64)
    for b in range(B):
        L = int(ctx_lens[b])
        T = int(tree_offsets[b + 1]) - int(tree_offsets[b])
        if T == 0:
            new_lens[b] = L
            continue
        n = int(n_accepted[b])
        nodes = [int(x) for x in path[b][:n]]
        if not (0 <= n <= T - 1) or any(not (0 < c < T) for c in nodes) or \
                any(nodes[i] >= nodes[i + 1] for i in range(n - 1)):
            raise ValueError(f"sequence {b}: path {nodes} is not increasing in (0, {T})")
        # read every source row before writing any destination: a destination
        # slot L+i can be the source slot of an earlier path entry
        def slot(t):
            return int(page_table[b][t // page_size]), t % page_size
        rows_k, rows_v = [], []
        for c in nodes:
            pg, off = slot(L + c)
            if layout == "NHD":
                rows_k.append(np.array(k_bits[pg, off])); rows_v.append(np.array(v_bits[pg, off]))
            else:
                rows_k.append(np.array(k_bits[pg, :, off])); rows_v.append(np.array(v_bits[pg, :, off]))
        for i, (rk, rv) in enumerate(zip(rows_k, rows_v), start=1):
            pg, off = slot(L + i)
            if layout == "NHD":
                k_out[pg, off] = rk; v_out[pg, off] = rv
            else:
                k_out[pg, :, off] = rk; v_out[pg, :, off] = rv
        new_lens[b] = L + 1 + n
    return k_out, v_out, new_lens


# --------------------------------------------------------------------------
# acceptance

def children_of(parents_local: Sequence[int], i: int) -> List[int]:
    """Children of node i in increasing node index."""
    return [c for c in range(len(parents_local)) if int(parents_local[c]) == i]


def greedy_accept(target_logits, draft_tokens, parents, tree_offsets):
    """Greedy walk: from the root, repeatedly move to the first child (lowest
    node index) whose draft token equals argmax of the current node's target
    logits (lowest token id on ties); stop when none does.  The bonus token is
    the argmax at the stop node.  Returns (paths, n_accepted, bonus) with
    local node indices."""
    target_logits = np.asarray(target_logits, dtype=np.float64)
    B = len(tree_offsets) - 1
    paths, n_acc, bonus = [], [], []
    for b in range(B):
        n0, n1 = int(tree_offsets[b]), int(tree_offsets[b + 1])
        if n1 == n0:
            paths.append([]); n_acc.append(0); bonus.append(-1)
            continue
        par = [int(x) for x in parents[n0:n1]]
        i, path = 0, []
        while True:
            y = int(np.argmax(target_logits[n0 + i]))   # first max = lowest id
            nxt = None
            for c in children_of(par, i):
                if int(draft_tokens[n0 + c]) == y:
                    nxt = c
                    break
            if nxt is None:
                break
            path.append(nxt)
            i = nxt
        paths.append(path)
        n_acc.append(len(path))
        bonus.append(int(np.argmax(target_logits[n0 + i])))
    return paths, n_acc, bonus


def softmax64(logits) -> np.ndarray:
    x = np.asarray(logits, dtype=np.float64)
    e = np.exp(x - x.max())
    return e / e.sum()


def inverse_cdf(p: np.ndarray, u: float) -> int:
    """Smallest x with sum_{y<=x} p_y > u * sum(p) (vocabulary order)."""
    c = np.cumsum(p)
    thr = u * c[-1]
    idx = int(np.searchsorted(c, thr, side="right"))
    return min(idx, len(p) - 1)


MUTATIONS = ("skip_accept", "resample_from_p", "unnormalised_residual",
             "wrong_uniform")


def rejection_accept(target_logits, draft_logits, draft_tokens, parents,
                     tree_offsets, uniforms, mutation: Optional[str] = None,
                     record: Optional[list] = None):
    """Exact tree rejection sampling (temperature 1).

    At node i with target p = softmax(target[i]) and draft q =
    softmax(draft[i]), the children c of i (drawn i.i.d. from q, tested in
    increasing node index) each propose x = draft_tokens[c]:
      accept iff uniforms[c, 0] * q(x) < p(x), i.e. u < min(1, p(x)/q(x));
      on rejection p <- max(0, p - q) / sum(max(0, p - q)) (kept if the sum
      is 0) and the next sibling is tested against the updated p.
    An accepted child becomes the current node; when no child is accepted
    (or i is a leaf) the bonus token is drawn from the current p by inverse
    CDF with uniforms[i, 1].

    `mutation` plants one of the known bugs (test-only): skip_accept,
    resample_from_p, unnormalised_residual, wrong_uniform.  `record`, if a
    list, receives one dict per decision with its margin |u - ratio| (the
    bonus draw's also carries u and the normalised CDF it was drawn from).
    """
    assert mutation is None or mutation in MUTATIONS
    target_logits = np.asarray(target_logits, dtype=np.float64)
    draft_logits = np.asarray(draft_logits, dtype=np.float64)
    uniforms = np.asarray(uniforms, dtype=np.float64)
    B = len(tree_offsets) - 1
    paths, n_acc, bonus = [], [], []
    for b in range(B):
        n0, n1 = int(tree_offsets[b]), int(tree_offsets[b + 1])
        if n1 == n0:
            paths.append([]); n_acc.append(0); bonus.append(-1)
            continue
        par = [int(x) for x in parents[n0:n1]]
        i, path = 0, []
        while True:
            p = softmax64(target_logits[n0 + i])
            q = softmax64(draft_logits[n0 + i])
            accepted = None
            for c in children_of(par, i):
                x = int(draft_tokens[n0 + c])
                u = uniforms[n0 + c, 1 if mutation == "wrong_uniform" else 0]
                if record is not None:
                    ratio = p[x] / q[x] if q[x] > 0 else math.inf
                    record.append(dict(seq=b, kind="accept", node=c,
                                       margin=abs(u - ratio)))
                if mutation == "skip_accept" or u * q[x] < p[x]:
                    accepted = c
                    break
                if mutation == "resample_from_p":
                    continue
                r = np.maximum(p - q, 0.0)
                z = r.sum()
                if z > 0:
                    p = r if mutation == "unnormalised_residual" else r / z
            if accepted is None:
                break
            path.append(accepted)
            i = accepted
        u1 = uniforms[n0 + i, 1]
        x = inverse_cdf(p, u1)
        if record is not None:
            c = np.cumsum(p)
            S = c[-1]
            lo = c[x - 1] / S if x > 0 else 0.0
            record.append(dict(seq=b, kind="bonus", node=i, u=u1, cdf=c / S,
                               margin=min(abs(u1 - lo), abs(u1 - c[x] / S))))
        paths.append(path)
        n_acc.append(len(path))
        bonus.append(x)
    return paths, n_acc, bonus
