"""GPU parity of ds_accept, through the C ABI.

Greedy: accepted paths, counts and bonus tokens bit-exact against the oracle.
Rejection: the same, except where the oracle's own decision margin
|u - p/q| (or, for the bonus draw, |u - CDF_x/S|) is below 1e-6: such a
sequence is compared up to that decision only, and each test allows at most
one such sequence.
"""
import numpy as np
import pytest
import torch

from long_context_speculative_ds_gb300 import binding as B
from long_context_speculative_ds_gb300 import synth
from oracle import ref
import helpers as H

pytestmark = pytest.mark.gpu


def _run_accept(step):
    step.accept()
    torch.cuda.synchronize()
    assert step.device_status() == 0
    n = step.out_n.cpu().numpy()
    paths = step.out_path.cpu().numpy()
    bonus = step.out_bonus.cpu().numpy()
    return [list(paths[b, :n[b]]) for b in range(len(n))], list(n), list(bonus), paths


def _check(st, inp, step, mode):
    """Returns (oracle paths, sequences exempted by a near-tie decision)."""
    g_paths, g_n, g_bonus, raw = _run_accept(step)
    for b in range(len(g_n)):
        assert (raw[b, g_n[b]:] == -1).all()
    tl = inp.target_logits.cpu().numpy()
    toks = inp.draft_tokens.cpu().numpy()
    if mode == "greedy":
        paths, n, bonus = ref.greedy_accept(tl, toks, st.parents, st.tree_offsets)
        assert g_paths == paths and g_n == n and g_bonus == bonus
        return paths, 0
    rec = []
    paths, n, bonus = ref.rejection_accept(
        tl, inp.draft_logits.cpu().numpy(), toks, st.parents, st.tree_offsets,
        inp.uniforms.cpu().numpy(), record=rec)
    exempt = H.check_rejection(g_paths, g_bonus, paths, bonus, rec, "rejection")
    return paths, exempt


@pytest.mark.parametrize("mode", ["greedy", "reject"])
def test_tiny_workload(mode):
    wl = synth.WORKLOADS["tiny"]
    st, inp, _ = H.build_case(wl, mode=mode)
    step = H.make_step(wl, inp, mode)
    assert _check(st, inp, step, mode)[1] <= 1


@pytest.mark.parametrize("mode", ["greedy", "reject"])
@pytest.mark.parametrize("vocab", [5, 256, 1001, 32000])
def test_many_random_trees(mode, vocab):
    """Batches of random trees (up to 64 nodes, duplicates among siblings
    allowed), vocabularies that are and are not multiples of 4."""
    wl = synth.tiny_workload(batch=12, vocab=vocab, max_depth=10, max_branch=4)
    accepted = exempt = 0
    for seed in range(4):
        rng = np.random.default_rng(seed)
        trees = [int(x) for x in rng.integers(1, 65, size=12)]
        trees[0] = 1
        st, inp, _ = H.build_case(wl, mode=mode, seed=100 + seed,
                                  ctx_lens=[32] * 12, tree_sizes=trees,
                                  draft="noisy")
        step = H.make_step(wl, inp, mode)
        paths, ex = _check(st, inp, step, mode)
        accepted += sum(len(p) for p in paths)
        exempt += ex
    assert accepted > 0    # the accept branch is exercised
    assert exempt <= 1


@pytest.mark.parametrize("mode", ["greedy", "reject"])
def test_vocabulary_beyond_the_register_slices(mode):
    """A vocabulary whose per-CTA slice exceeds what the rejection node pass
    holds in registers and shared memory (here 200,000 > 163,840 tokens) takes
    the streaming node pass; greedy runs its usual argmax pass."""
    wl = synth.tiny_workload(batch=3, vocab=200000, max_depth=6, max_branch=3)
    st, inp, _ = H.build_case(wl, mode=mode, seed=7, ctx_lens=[32] * 3,
                              tree_sizes=[9, 1, 14], draft="noisy")
    step = H.make_step(wl, inp, mode)
    assert _check(st, inp, step, mode)[1] <= 1


def test_one_hot_target_rejection_equals_greedy():
    wl = synth.tiny_workload(batch=6, vocab=300, max_depth=6, max_branch=3)
    st, inp, _ = H.build_case(wl, mode="reject", seed=21,
                              ctx_lens=[16] * 6, tree_sizes=[10, 20, 1, 33, 64, 7])
    tl = inp.target_logits
    am = tl.argmax(dim=1)
    hot = tl.clone()
    hot[torch.arange(tl.shape[0], device=tl.device), am] += 1e4
    # make the first child of each node carry its parent's argmax
    toks = inp.draft_tokens.clone()
    seen = set()
    for b in range(wl.batch):
        n0 = st.tree_offsets[b]
        for j in range(1, st.tree_sizes[b]):
            p = st.parents[n0 + j]
            if (b, p) not in seen:
                seen.add((b, p))
                toks[n0 + j] = am[n0 + p]
    inp.target_logits = hot
    inp.draft_tokens = toks
    rej = H.make_step(wl, inp, "reject")
    r = _run_accept(rej)
    greedy = H.make_step(wl, inp, "greedy")
    g = _run_accept(greedy)
    assert r[0] == g[0] and r[2] == g[2]
    assert sum(r[1]) > 0


@pytest.mark.parametrize("name,mode", [("llama8b-32k", "greedy"),
                                       ("llama8b-64k", "reject"),
                                       ("llama8b-128k-32l", "greedy"),
                                       ("qwen3-8b-ragged-b8", "reject")])
def test_full_size(name, mode):
    wl = synth.WORKLOADS[name]
    st, inp, _ = H.build_case(wl, layers=1, mode=mode)
    step = H.make_step(wl, inp, mode)
    assert _check(st, inp, step, mode)[1] <= 1
