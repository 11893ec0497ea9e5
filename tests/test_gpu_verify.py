"""GPU parity of ds_verify_attn against the float64 oracle, through the C ABI.

Bars: attention output |gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise; chunk
scores within 1e-3 relative.  Small cases span several key tiles, ragged
tails, empty contexts, single nodes, chains, all supported head dims, page
sizes, chunk sizes, group sizes (including two row groups) and both cache
layouts; the four large workloads run at full size for one layer here, and
the headline and ragged workloads run as whole multi-layer steps (summed
scores, retrieval, acceptance) in test_gpu_fullstep.py.
"""
import math

import numpy as np
import pytest
import torch

from long_context_speculative_ds_gb300 import binding as B
from long_context_speculative_ds_gb300 import synth
from oracle import ref
import helpers as H

pytestmark = pytest.mark.gpu


def _run_verify(wl, st, inp, mode, layout="NHD", out_dtype=torch.bfloat16,
                layers=1, **kw):
    step = H.make_step(wl, inp, mode, layout, out_dtype, **kw)
    for l in range(layers):
        step.verify_layer(l)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    return step


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_tiny_workload(layout, out_dtype):
    wl = synth.WORKLOADS["tiny"]
    st, inp, mode = H.build_case(wl, layout=layout)
    step = _run_verify(wl, st, inp, mode, layout, out_dtype)
    o, s, _ = H.oracle_layer(wl, st, inp, 0, layout, step.max_chunks)
    H.assert_attention_close(step.out[0], o, "tiny out")
    H.assert_scores_close(step.scores, s, st, wl, "tiny scores")


EDGE = [
    # (name, overrides, ctx_lens, tree_sizes)
    ("ragged_b3", dict(batch=3), (300, 0, 77), (8, 5, 1)),
    ("tile_edges", dict(batch=2), (128, 256 - 3), (3, 3)),
    ("chain64", dict(batch=1, max_depth=64, max_branch=1), (200,), (64,)),
    ("star64", dict(batch=1, max_depth=1, max_branch=64), (129,), (64,)),
    ("d128_g4", dict(batch=2, num_q_heads=16, num_kv_heads=4, head_dim=128,
                     chunk_size=64), (1000, 333), (30, 17)),
    ("g8_two_rowgroups", dict(batch=1, num_q_heads=16, num_kv_heads=2,
                              head_dim=128, chunk_size=16), (500,), (64,)),
    ("g1", dict(batch=2, num_q_heads=2, num_kv_heads=2), (64, 190), (9, 2)),
    ("page32_chunk128", dict(batch=2, page_size=32, chunk_size=128), (700, 31),
     (12, 4)),
    ("g16", dict(batch=1, num_q_heads=16, num_kv_heads=1), (96,), (20,)),
]


@pytest.mark.parametrize("name,over,ctx,trees", EDGE, ids=[e[0] for e in EDGE])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_edge_cases(name, over, ctx, trees, layout):
    wl = synth.tiny_workload(window=64, top_k=2, **over)
    st, inp, mode = H.build_case(wl, layout=layout, ctx_lens=ctx,
                                 tree_sizes=trees, seed=sum(map(ord, name)))
    step = _run_verify(wl, st, inp, mode, layout, torch.float32)
    o, s, tmass = H.oracle_layer(wl, st, inp, 0, layout, step.max_chunks)
    H.assert_attention_close(step.out[0], o, name)
    H.assert_scores_close(step.scores, s, st, wl, name)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_accumulate_over_layers_and_untouched_tail(layout):
    """Layers after the first plan their work and fetch their first
    context tile before the preceding kernel has finished."""
    wl = synth.tiny_workload(batch=2, layers=3)
    st, inp, mode = H.build_case(wl, layers=3, ctx_lens=(150, 40), layout=layout,
                                 tree_sizes=(6, 3), seed=5)
    step = H.make_step(wl, inp, mode, layout)
    step.scores.fill_(7.0)           # overwritten by layer 0, then summed
    step.run()
    torch.cuda.synchronize()
    total = 0
    for l in range(3):
        o, s, _ = H.oracle_layer(wl, st, inp, l, layout, step.max_chunks)
        H.assert_attention_close(step.out[l], o, f"layer {l}")
        total = total + s
    H.assert_scores_close(step.scores, total, st, wl, "summed")
    # entries beyond each sequence's chunk count keep their old value
    g = step.scores.cpu().numpy()
    assert (g[1, -(-40 // wl.chunk_size):] == 7.0).all()


def test_many_small_sms():
    """A tiny num_sms forces long splits; a huge one forces one tile each."""
    wl = synth.tiny_workload(batch=2)
    for sms in (1, 3, 1000):
        st, inp, mode = H.build_case(wl, ctx_lens=(900, 260), tree_sizes=(8, 7),
                                     seed=sms)
        step = _run_verify(wl, st, inp, mode, num_sms=sms)
        o, s, _ = H.oracle_layer(wl, st, inp, 0, "NHD", step.max_chunks)
        H.assert_attention_close(step.out[0], o, f"sms={sms}")
        H.assert_scores_close(step.scores, s, st, wl, f"sms={sms}")


def test_plan_fitted_to_the_ctas():
    """Per-sequence rounding of the split count overflows the CTAs here (14
    items at 7 tiles per split for 12 CTAs), so the plan refits to 8 tiles
    per split and 12 items; two layers, the second accumulating scores
    (its plan is formed before the wait on the preceding kernel)."""
    wl = synth.tiny_workload(batch=4, layers=2)
    st, inp, mode = H.build_case(wl, layers=2, ctx_lens=(300, 2000, 700, 1500),
                                 tree_sizes=(5, 9, 3, 7), seed=12)
    step = _run_verify(wl, st, inp, mode, layers=2, num_sms=12)
    total = 0
    for l in range(2):
        o, s, _ = H.oracle_layer(wl, st, inp, l, "NHD", step.max_chunks)
        H.assert_attention_close(step.out[l], o, f"refit layer {l}")
        total = total + s
    H.assert_scores_close(step.scores, total, st, wl, "refit summed")


@pytest.mark.parametrize("sms", [0, 1000])
def test_sequence_without_tree_nodes(sms):
    """A sequence with no tree nodes has no work item: its chunks get zero
    scores (entries past a sequence's chunks keep their old value), next to
    sequences that do have trees, with the device's CTAs and with 1000
    planned CTAs (one tile per item)."""
    wl = synth.tiny_workload(batch=3)
    st, inp, mode = H.build_case(wl, ctx_lens=(600, 300, 200), tree_sizes=(5, 0, 7),
                                 seed=31)
    step = H.make_step(wl, inp, mode, num_sms=sms)
    step.scores.fill_(7.0)
    step.verify_layer(0)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    o, s, _ = H.oracle_layer(wl, st, inp, 0, "NHD", step.max_chunks)
    H.assert_attention_close(step.out[0], o, f"sms={sms}")
    H.assert_scores_close(step.scores, s, st, wl, f"sms={sms}")
    g = step.scores.cpu().numpy()
    n1 = -(-300 // wl.chunk_size)
    assert (g[1, :n1] == 0.0).all()
    assert (g[1, n1:] == 7.0).all() and (g[2, -(-200 // wl.chunk_size):] == 7.0).all()


@pytest.mark.parametrize("name", ["llama8b-32k", "llama8b-64k",
                                  "llama8b-128k-32l", "qwen3-8b-ragged-b8"])
def test_full_size_one_layer(name):
    wl = synth.WORKLOADS[name]
    st, inp, mode = H.build_case(wl, layers=1)
    step = _run_verify(wl, st, inp, mode)
    o, s, tmass = H.oracle_layer(wl, st, inp, 0, "NHD", step.max_chunks)
    H.assert_attention_close(step.out[0], o, name)
    H.assert_scores_close(step.scores, s, st, wl, name)
    # mass invariant on the GPU's own scores: sum + tree mass = T * H_q
    g = step.scores.double().cpu().numpy()
    for b in range(wl.batch):
        want = st.tree_sizes[b] * wl.num_q_heads - tmass[b]
        assert abs(g[b].sum() - want) <= 1e-4 * st.tree_sizes[b] * wl.num_q_heads
