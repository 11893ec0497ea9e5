"""Whole verify steps at full size against the float64 oracle, through the C ABI.

The headline workload (Llama-3.1-8B KV shapes, 128K context, 64-node tree)
and the ragged batch-8 serving workload run as the benchmark runs them:
several layers of verify attention with the chunk salience summed over the
layers, then top-k chunk selection plus window gathered into the compact
cache with the workload's local RoPE, then acceptance (vllm-diffspec README,
"What DiffSpec Does", last paragraph: chunks plus a rolling window rebuilt
as a compact cache; "Key Results": Llama-3.1-8B at 128K).

Checked: every layer's output (2e-3 + 1e-2 |ref|), the summed scores
(1e-3 relative) and their mass invariant, the selection bit-exact against
the oracle's rule on the GPU's own summed scores and against the float64
selection up to near-ties, every planted chunk chosen, the compact cache
(ids, lengths, positions and V byte-exact, K under the RoPE tolerance), and
the accepted path and bonus.

The headline runs 4 of its 32 layers (the layers differ only in their seeds,
so 4 cover the accumulation as well as 32 would); the ragged workload runs
2 of its 36.
"""
import numpy as np
import pytest
import torch

from long_context_speculative_ds_gb300 import synth
from oracle import ref
import helpers as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,layers", [("llama8b-128k-32l", 4),
                                         ("qwen3-8b-ragged-b8", 2)])
def test_whole_step(name, layers):
    wl = synth.WORKLOADS[name].replace(layers=layers)
    st, inp, mode = H.build_case(wl, layers=layers)
    step = H.make_step(wl, inp, mode, rope_base=wl.rope_base)
    step.run()
    torch.cuda.synchronize()
    assert step.device_status() == 0

    total, tmass_total = 0.0, 0.0
    for l in range(layers):
        o, s, tmass = H.oracle_layer(wl, st, inp, l, "NHD", step.max_chunks)
        H.assert_attention_close(step.out[l], o, f"{name} layer {l}")
        total = total + s
        tmass_total = tmass_total + np.asarray(tmass)
    H.assert_scores_close(step.scores, total, st, wl, f"{name} summed scores")
    g = step.scores.double().cpu().numpy()
    for b in range(wl.batch):
        want = layers * st.tree_sizes[b] * wl.num_q_heads - tmass_total[b]
        scale = layers * st.tree_sizes[b] * wl.num_q_heads
        assert abs(g[b].sum() - want) <= 1e-4 * scale

    # retrieval: the oracle's rule on the GPU's scores, byte for byte
    H.check_gather(wl, st, inp, step, g, "NHD", rope_base=wl.rope_base)
    H.check_selection_vs_f64(wl, st, g, total)

    # acceptance
    tl = inp.target_logits.cpu().numpy()
    toks = inp.draft_tokens.cpu().numpy()
    n = step.out_n.cpu().numpy()
    paths = step.out_path.cpu().numpy()
    g_paths = [list(paths[b, :n[b]]) for b in range(wl.batch)]
    g_bonus = list(step.out_bonus.cpu().numpy())
    if mode == "greedy":
        rp, _, rb = ref.greedy_accept(tl, toks, st.parents, st.tree_offsets)
        assert g_paths == rp and g_bonus == rb
    else:
        rec = []
        rp, _, rb = ref.rejection_accept(tl, inp.draft_logits.cpu().numpy(), toks,
                                         st.parents, st.tree_offsets,
                                         inp.uniforms.cpu().numpy(), record=rec)
        assert H.check_rejection(g_paths, g_bonus, rp, rb, rec, name) <= 1
