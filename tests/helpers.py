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
