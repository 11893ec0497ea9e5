"""Pins of the oracle's compact-cache append (oracle.ref.compact_append).

Between retrievals the compact cache is kept and only the newly committed
tokens are appended (vllm-diffspec README, "What DiffSpec Does" item 4;
"Configuration", diffspec_retrieval_interval).  Pinned against the gather
oracle: with no chunks selected and a window covering everything, gathering
L1 tokens and appending [L1, L2) must equal gathering L2 tokens outright,
with and without the local RoPE (the local positions coincide); plus the
refusal of rows that do not fit and the empty append.
"""
import numpy as np
import pytest

from oracle import ref

P, H, D = 16, 2, 64


def _case(rng, L2):
    pages = (L2 + P - 1) // P + 2
    pt = np.array([rng.permutation(pages)])
    bits = lambda: ((rng.standard_normal((pages, P, H, D)).astype(np.float32)).view(np.uint32)
                    >> 16).astype(np.uint16)
    return pt, bits(), bits()


@pytest.mark.parametrize("rope", [0.0, 10000.0])
def test_append_equals_full_window_gather(rope):
    rng = np.random.default_rng(7)
    L1, L2 = 150, 171
    pt, k, v = _case(rng, L2)
    cap = 256
    kw = dict(page_size=P, chunk_size=32, top_k=0, window=cap, capacity=cap, rope_base=rope)
    scores = np.zeros((1, 16))
    first = ref.gather_compact(k, v, pt, [L1], scores, **kw)
    inc = ref.compact_append(first, k, v, pt, [L1], [L2], P, rope_base=rope)
    full = ref.gather_compact(k, v, pt, [L2], scores, **kw)
    assert inc["out_len"].tolist() == [L2]
    for key in ("positions", "out_k", "out_v"):
        np.testing.assert_array_equal(inc[key][0, :L2], full[key][0, :L2])


def test_append_refuses_overflow_and_keeps_rows():
    rng = np.random.default_rng(8)
    pt, k, v = _case(rng, 100)
    kw = dict(page_size=P, chunk_size=32, top_k=0, window=64, capacity=64)
    first = ref.gather_compact(k, v, pt, [60], np.zeros((1, 8)), **kw)
    same = ref.compact_append(first, k, v, pt, [60], [80], P)        # 64 + 20 > 64
    for key in first:
        np.testing.assert_array_equal(same[key], first[key])
    none = ref.compact_append(first, k, v, pt, [60], [60], P)
    assert none["out_len"].tolist() == first["out_len"].tolist()
