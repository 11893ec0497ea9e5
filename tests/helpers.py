"""Shared helpers of the GPU parity tests: build seeded inputs, run the
library through the C ABI, and run the float64 oracle on the same values."""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np
import torch

from long_context_speculative_ds_gb300 import binding as B
from long_context_speculative_ds_gb300 import synth
from long_context_speculative_ds_gb300.step import StepInputs, VerifyStep
from oracle import ref

ATOL_O, RTOL_O = 2e-3, 1e-2        # attention output bar
RTOL_SCORE = 1e-3                  # chunk-score bar
EXEMPT = 1e-6                      # rejection-draw exemption |u - ratio|


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def build_case(wl: synth.Workload, *, layers: int = 1, layout: str = "NHD",
               mode: Optional[str] = None, seed: Optional[int] = None,
               ctx_lens=None, tree_sizes=None, parents=None, device="cuda",
               draft: Optional[str] = None, plant: bool = True):
    st = synth.make_structure(wl, seed=seed, ctx_lens=ctx_lens,
                              tree_sizes=tree_sizes, parents=parents)
    dev = torch.device(device)
    qs, ks, vs = [], [], []
    for l in range(layers):
        q, k, v = synth.make_layer(st, l, device=dev, layout=layout,
                                   seed=None if seed is None else seed + 10 + l,
                                   plant=plant)
        qs.append(q); ks.append(k); vs.append(v)
    sk, sv = synth.make_source_cache(st, device=dev, layout=layout,
                                     seed=None if seed is None else seed + 999)
    mode = mode or ("reject" if wl.accept == "reject" else "greedy")
    acc = synth.make_accept_inputs(st, mode, device=dev,
                                   seed=None if seed is None else seed + 500,
                                   draft=draft)
    i32 = dict(dtype=torch.int32, device=dev)
    inp = StepInputs(
        page_table=st.page_table.to(dev),
        ctx_lens=torch.tensor(st.ctx_lens, **i32),
        tree_offsets=torch.tensor(st.tree_offsets, **i32),
        parents=torch.tensor(st.parents, **i32) if st.n_nodes else torch.zeros(1, **i32),
        q=qs, k_cache=ks, v_cache=vs, src_k=sk, src_v=sv,
        target_logits=acc.target_logits, draft_logits=acc.draft_logits,
        draft_tokens=acc.draft_tokens, uniforms=acc.uniforms)
    return st, inp, mode


def make_step(wl, inp, mode, layout="NHD", out_dtype=torch.bfloat16, **kw):
    return VerifyStep(inp, chunk_size=wl.chunk_size, top_k=wl.top_k,
                      window=wl.window, accept_mode=mode, kv_layout=layout,
                      out_dtype=out_dtype, **kw)


def oracle_layer(wl, st, inp, l, layout="NHD", max_chunks=None):
    return ref.verify_attention(
        f64(inp.q[l]), f64(inp.k_cache[l]), f64(inp.v_cache[l]),
        st.page_table.numpy(), st.ctx_lens, st.tree_offsets, st.parents,
        wl.page_size, wl.chunk_size, layout=layout, max_chunks=max_chunks)


def assert_attention_close(gpu: torch.Tensor, ref_o: np.ndarray, what=""):
    g = f64(gpu)
    err = np.abs(g - ref_o)
    bound = ATOL_O + RTOL_O * np.abs(ref_o)
    bad = err > bound
    assert not bad.any(), (
        f"{what}: {int(bad.sum())} of {bad.size} outside 2e-3 + 1e-2|ref|;"
        f" max abs err {err.max():.3e}")
    return float(err.max())


def assert_scores_close(gpu: torch.Tensor, ref_s: np.ndarray, st, wl, what=""):
    g = f64(gpu)
    worst = 0.0
    for b in range(len(st.ctx_lens)):
        n = -(-st.ctx_lens[b] // wl.chunk_size)
        gg, rr = g[b, :n], ref_s[b, :n]
        rel = np.abs(gg - rr) / np.maximum(np.abs(rr), 1e-30)
        assert (rel <= RTOL_SCORE).all(), (
            f"{what}: seq {b} chunk scores rel err {rel.max():.3e}")
        worst = max(worst, float(rel.max()) if n else 0.0)
    return worst


def check_rejection(g_paths, g_bonus, paths, bonus, rec, what=""):
    """Rejection draws of the GPU against the oracle's, decision by decision.

    Accept tests: a sequence is compared in full unless one of its accept
    tests has a margin |u - p/q| below EXEMPT; then only what precedes that
    test is compared (the accepted nodes before it must open the GPU's path).
    Such sequences are returned as the count the tests bound.

    Bonus draws: when u lies within EXEMPT of a boundary of the inverse CDF
    (frequent at large vocabularies, where the CDF steps are a few 1e-6
    apart) the whole path must still match and the GPU's token must be one
    whose CDF interval [CDF(x-1), CDF(x)) comes within EXEMPT of u; those
    sequences are reported but not counted."""
    by_seq = {}
    for r in rec:
        by_seq.setdefault(r["seq"], []).append(r)
    exempt = bonus_ties = 0
    for b in range(len(paths)):
        rs = by_seq.get(b, [])
        tie = next((k for k, r in enumerate(rs) if r["margin"] < EXEMPT), None)
        if tie is None:
            assert list(g_paths[b]) == list(paths[b]) and g_bonus[b] == bonus[b], \
                f"{what}: sequence {b}: gpu {g_paths[b]}/{g_bonus[b]}, " \
                f"oracle {paths[b]}/{bonus[b]}"
            continue
        r = rs[tie]
        if r["kind"] == "bonus":
            bonus_ties += 1
            assert list(g_paths[b]) == list(paths[b]), f"{what}: sequence {b}"
            x, cdf, u = int(g_bonus[b]), r["cdf"], r["u"]
            assert 0 <= x < len(cdf), f"{what}: sequence {b}: bonus {x}"
            lo = cdf[x - 1] if x > 0 else 0.0
            assert lo - EXEMPT <= u < cdf[x] + EXEMPT, \
                f"{what}: sequence {b}: bonus {x} outside the near-tie of u"
            continue
        exempt += 1
        on_path = set(paths[b])
        prefix = [q["node"] for q in rs[:tie] if q["kind"] == "accept"
                  and q["node"] in on_path]
        assert list(g_paths[b][:len(prefix)]) == prefix, f"{what}: sequence {b}"
    print(f"{what}: {exempt} of {len(paths)} sequences with an accept test "
          f"within {EXEMPT} of its threshold, {bonus_ties} with a bonus draw "
          f"within {EXEMPT} of a CDF boundary (checked for validity)")
    return exempt


def check_gather(wl, st, inp, step, scores_np, layout="NHD", rope_base=0.0):
    """Compact cache of the GPU against the oracle's gather on the same
    scores: chunk ids, lengths, positions and V byte-exact; K byte-exact
    without RoPE; with RoPE within ulp_bf16(ref) + 1e-6 |pair| of the
    oracle's once-rounded float64 rotation (the kernel's angle error scales
    with the pair's norm before the rounding to bf16) and >= 99.5 % equal."""
    exp = ref.gather_compact(bits(inp.src_k), bits(inp.src_v),
                             st.page_table.numpy(), st.ctx_lens, scores_np,
                             wl.page_size, wl.chunk_size, wl.top_k, wl.window,
                             step.capacity, layout=layout, rope_base=rope_base)
    ids = step.out_chunk_ids.cpu().numpy()[:, :wl.top_k]
    np.testing.assert_array_equal(ids, exp["chunk_ids"])
    np.testing.assert_array_equal(step.out_len.cpu().numpy(), exp["out_len"])
    np.testing.assert_array_equal(step.out_positions.cpu().numpy(),
                                  exp["positions"])
    ok, ov = bits(step.out_k), bits(step.out_v)
    exact = total = 0
    for b in range(wl.batch):
        n = exp["out_len"][b]
        np.testing.assert_array_equal(ov[b, :n], exp["out_v"][b, :n])
        if rope_base == 0.0:
            np.testing.assert_array_equal(ok[b, :n], exp["out_k"][b, :n])
            continue
        g = ref.bf16_bits_to_f64(ok[b, :n])
        o = ref.bf16_bits_to_f64(exp["out_k"][b, :n])
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o), 1e-30))) - 7)
        half = wl.head_dim // 2
        pair = np.sqrt(o[..., :half] ** 2 + o[..., half:] ** 2)
        pair = np.concatenate([pair, pair], axis=-1)
        err = np.abs(g - o)
        assert (err <= ulp + 1e-6 * pair).all(), f"seq {b}: max err {err.max()}"
        exact += int((ok[b, :n] == exp["out_k"][b, :n]).sum())
        total += ok[b, :n].size
    if rope_base != 0.0:
        assert exact >= 0.995 * total, (exact, total)
    return exp


def check_selection_vs_f64(wl, st, gpu_scores, f64_scores):
    """The GPU's selection (made from its own scores) against the selection
    from float64 oracle scores: any difference must be a near-tie,
    |s_k - s_(k+1)| <= 1e-3 s_k, and every planted chunk must be chosen."""
    for b in range(wl.batch):
        L = st.ctx_lens[b]
        got = ref.select_chunks(gpu_scores[b], L, wl.chunk_size, wl.top_k, wl.window)
        want = ref.select_chunks(f64_scores[b], L, wl.chunk_size, wl.top_k, wl.window)
        if got != want:
            n = ref.candidate_count(L, wl.chunk_size, wl.window)
            srt = np.sort(f64_scores[b, :n])[::-1]
            sk, sk1 = srt[wl.top_k - 1], srt[wl.top_k]
            assert abs(sk - sk1) <= 1e-3 * sk, \
                f"seq {b}: selection differs beyond a near-tie"
        assert set(st.planted_chunks[b]) <= set(got), \
            f"seq {b}: a planted chunk was missed"
