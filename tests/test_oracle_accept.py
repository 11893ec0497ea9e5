"""Pins for the oracle's greedy and rejection acceptance (CPU only).

* greedy: brute force over every root-to-leaf path; the chain case is the
  textbook longest matching prefix; rejection with one-hot targets
  (temperature -> 0) reproduces greedy (adaptive-specdec README, "Correctness
  first", G2: greedy is not special-cased).
* rejection: the emitted tokens must follow the exact autoregressive marginal
  of a tiny enumerable model (same README, G1: total variation below 0.02
  and a chi-square test), every planted bug must fail that gate, and the
  single-candidate acceptance rate must equal 1 - TV(p, q) (same README,
  "The controller").
"""
import json
import math
import os

import numpy as np
import pytest
from scipy import stats

from oracle import brute, ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _random_tree(rng, T, branch=3):
    par = [-1]
    nch = [0]
    for j in range(1, T):
        ok = [i for i in range(j) if nch[i] < branch]
        p = int(rng.choice(ok))
        par.append(p)
        nch.append(0)
        nch[p] += 1
    return par


@pytest.mark.parametrize("seed", range(20))
def test_greedy_matches_path_brute_force(seed):
    rng = np.random.default_rng(seed)
    T, V = int(rng.integers(1, 12)), 6
    par = _random_tree(rng, T)
    logits = rng.integers(0, 3, size=(T, V)).astype(np.float64)  # ties
    tokens = np.zeros(T, dtype=np.int64)
    # distinct tokens among siblings, biased toward the parent's argmax
    for i in range(T):
        kids = [c for c in range(T) if par[c] == i]
        toks = rng.permutation(V)[:len(kids)]
        if kids and rng.random() < 0.7:
            am = int(np.argmax(logits[i]))
            toks = [am] + [t for t in rng.permutation(V) if t != am][:len(kids) - 1]
        for c, t in zip(kids, toks):
            tokens[c] = t
    paths, n_acc, bonus = ref.greedy_accept(logits, tokens, par, [0, T])
    bp, bb = brute.greedy_by_paths(logits, tokens, par)
    assert paths[0] == bp and n_acc[0] == len(bp) and bonus[0] == bb


def test_greedy_chain_is_longest_matching_prefix():
    rng = np.random.default_rng(5)
    T, V = 9, 5
    par = [-1] + list(range(T - 1))
    for _ in range(50):
        logits = rng.normal(size=(T, V))
        tokens = rng.integers(0, V, size=T)
        am = np.argmax(logits, axis=1)
        # textbook: count matches of draft[j+1] with target argmax at j
        n = 0
        while n + 1 < T and tokens[n + 1] == am[n]:
            n += 1
        paths, n_acc, bonus = ref.greedy_accept(logits, tokens, par, [0, T])
        assert n_acc[0] == n
        assert paths[0] == list(range(1, n + 1))
        assert bonus[0] == am[n]


def test_greedy_tie_rules():
    """Argmax ties go to the lower token id; duplicate sibling tokens go to
    the lower node index."""
    logits = np.array([[0., 5., 5.], [1., 0., 0.], [0., 0., 2.], [3., 0., 0.]])
    tokens = np.array([0, 1, 1, 2])
    par = [-1, 0, 0, 1]
    paths, n_acc, bonus = ref.greedy_accept(logits, tokens, par, [0, 4])
    # root argmax = 1 (tie 1/2 -> 1); children 1 and 2 both carry 1 -> node 1;
    # node 1 argmax = 0, child 3 carries 2 -> stop; bonus = argmax(node 1) = 0
    assert paths[0] == [1] and bonus[0] == 0


def test_golden_worked_greedy():
    with open(os.path.join(GOLDEN, "greedy_worked.json")) as f:
        g = json.load(f)
    paths, n_acc, bonus = ref.greedy_accept(
        np.array(g["target_logits"]), g["draft_tokens"], g["parents"],
        g["tree_offsets"])
    assert paths == g["expect_paths"]
    assert n_acc == g["expect_n_accepted"]
    assert bonus == g["expect_bonus"]


def test_rejection_with_one_hot_target_is_greedy():
    rng = np.random.default_rng(11)
    for _ in range(40):
        T, V = int(rng.integers(1, 10)), 7
        par = _random_tree(rng, T)
        tl = rng.normal(size=(T, V))
        hot = tl.copy()
        hot[np.arange(T), np.argmax(tl, axis=1)] += 1e4   # exp(-1e4) == 0
        dl = rng.normal(size=(T, V))
        tokens = rng.integers(0, V, size=T)
        for i in range(T):
            kids = [c for c in range(T) if par[c] == i]
            if kids and rng.random() < 0.6:
                tokens[kids[int(rng.integers(len(kids)))]] = np.argmax(tl[i])
        u = rng.random((T, 2))
        g = ref.greedy_accept(tl, tokens, par, [0, T])
        r = ref.rejection_accept(hot, dl, tokens, par, [0, T], u)
        assert g == r


# ---------------------------------------------------------------------------
# G1: distributional equivalence on an enumerable model

V_SMALL = 8


class TinyModel:
    """Target and draft next-token logits for every prefix of length <= 2."""

    def __init__(self, seed):
        rng = np.random.default_rng(seed)
        self.t = {(): rng.normal(0, math.sqrt(2), V_SMALL)}
        for a in range(V_SMALL):
            self.t[(a,)] = rng.normal(0, math.sqrt(2), V_SMALL)
        self.d = {k: v + rng.normal(0, 1, V_SMALL) for k, v in self.t.items()}
        self.p = {k: ref.softmax64(v) for k, v in self.t.items()}
        self.q = {k: ref.softmax64(v) for k, v in self.d.items()}

    def exact_joint(self):
        j = np.zeros((V_SMALL, V_SMALL))
        for a in range(V_SMALL):
            j[a] = self.p[()][a] * self.p[(a,)]
        return j


def _draw(rng, probs):
    return int(np.searchsorted(np.cumsum(probs), rng.random() * probs.sum(),
                               side="right").clip(0, len(probs) - 1))


def _emit_pairs(model, n_runs, seed, mutation=None, branch=(1, 3), sub=(0, 2)):
    """Run the oracle walk n_runs times on freshly drawn trees (depth <= 2);
    return counts over the first two emitted tokens (continuing
    autoregressively from the exact target when only one token came out)."""
    rng = np.random.default_rng(seed)
    counts = np.zeros((V_SMALL, V_SMALL), dtype=np.int64)
    for _ in range(n_runs):
        par, toks, pref = [-1], [0], [()]
        for _c in range(int(rng.integers(branch[0], branch[1] + 1))):
            a = _draw(rng, model.q[()])
            par.append(0); toks.append(a); pref.append((a,))
        n1 = len(par)
        for c in range(1, n1):
            a = toks[c]
            for _g in range(int(rng.integers(sub[0], sub[1] + 1))):
                # the logits after a depth-2 prefix are never read for the
                # first two tokens; reuse the depth-1 row as a placeholder
                b = _draw(rng, model.q[(a,)])
                par.append(c); toks.append(b); pref.append((a, b))
        T = len(par)
        tl = np.stack([model.t[p if len(p) < 2 else p[:1]] for p in pref])
        dl = np.stack([model.d[p if len(p) < 2 else p[:1]] for p in pref])
        u = rng.random((T, 2))
        paths, n_acc, bonus = ref.rejection_accept(tl, dl, toks, par, [0, T],
                                                   u, mutation=mutation)
        emitted = [toks[c] for c in paths[0]] + [bonus[0]]
        if len(emitted) < 2:
            emitted.append(_draw(rng, model.p[(emitted[0],)]))
        counts[emitted[0], emitted[1]] += 1
    return counts


def _tv_and_p(counts, joint):
    n = counts.sum()
    emp = counts / n
    tv = 0.5 * np.abs(emp - joint).sum()
    chi = stats.chisquare(counts.ravel(), joint.ravel() * n)
    return tv, chi.pvalue


def test_g1_emitted_tokens_follow_exact_ar_marginal():
    model = TinyModel(3)
    counts = _emit_pairs(model, 200000, seed=1)
    tv, pval = _tv_and_p(counts, model.exact_joint())
    floor = math.sqrt(V_SMALL * V_SMALL / (2 * math.pi * counts.sum()))
    assert tv < 0.02, (tv, floor)
    assert pval > 0.01, pval


@pytest.mark.parametrize("mutation", ref.MUTATIONS)
def test_g1_catches_each_planted_bug(mutation):
    model = TinyModel(3)
    counts = _emit_pairs(model, 20000, seed=2, mutation=mutation)
    tv, pval = _tv_and_p(counts, model.exact_joint())
    # the gate of the correct walk is (tv < 0.02 and pval > 0.01); each bug
    # must fail it decisively
    assert tv >= 0.02 or pval < 1e-6, (mutation, tv, pval)
    assert pval < 1e-6, (mutation, tv, pval)


def test_single_candidate_acceptance_is_one_minus_tv():
    model = TinyModel(4)
    p, q = model.p[()], model.q[()]
    rng = np.random.default_rng(9)
    n, acc = 40000, 0
    tl = np.stack([model.t[()], model.t[()]])
    dl = np.stack([model.d[()], model.d[()]])
    for _ in range(n):
        x = _draw(rng, q)
        u = rng.random((2, 2))
        paths, _, _ = ref.rejection_accept(tl, dl, [0, x], [-1, 0], [0, 2], u)
        acc += len(paths[0])
    expect = np.minimum(p, q).sum()
    assert abs(expect - (1 - 0.5 * np.abs(p - q).sum())) < 1e-12
    sd = math.sqrt(expect * (1 - expect) / n)
    assert abs(acc / n - expect) < 4 * sd


def test_golden_acceptance_identity():
    with open(os.path.join(GOLDEN, "acceptance_identity.json")) as f:
        g = json.load(f)
    p, q = np.array(g["p"]), np.array(g["q"])
    assert abs(np.minimum(p, q).sum() - g["expect_acceptance"]) < 1e-12
    assert abs(0.5 * np.abs(p - q).sum() - g["expect_tv"]) < 1e-12
    # the oracle's accept test on each token reproduces min(1, p/q)
    for x in range(len(p)):
        for u in (0.0, 0.25, 0.5, 0.999):
            _, n_acc, _ = ref.rejection_accept(
                np.log(np.stack([p, p])), np.log(np.stack([q, q])), [0, x],
                [-1, 0], [0, 2], np.array([[0.5, 0.5], [u, 0.5]]))
            assert n_acc[0] == (1 if u * q[x] < p[x] else 0)
