"""Pins of the oracle's RoPE rebuild of the compact cache (oracle.ref
rope_rotate, f64_to_bf16_bits and gather_compact with rope_base > 0).

The compact draft cache is rebuilt from pre-RoPE K with local positions
(vllm-diffspec README, "Architecture", dual-view draft cache).  Pinned
against: an independent float32 round-to-nearest-even on bit patterns, exact
ties, position 0 being the identity, the two-dimensional case being a plain
rotation by pos radians, pair norms being preserved, and the defining
property that rotated dot products depend only on the position difference.
"""
import math

import numpy as np
import pytest

from oracle import ref


def _rne_f32_bits(x32):
    """float32 -> bf16 by the usual integer trick (independent of frexp)."""
    u = np.asarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def test_rounding_matches_float32_rne():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * 10.0 ** rng.integers(-5, 5, 200000)).astype(np.float32)
    assert (ref.f64_to_bf16_bits(x.astype(np.float64)) == _rne_f32_bits(x)).all()


def test_rounding_ties_to_even():
    one = 1.0
    assert ref.f64_to_bf16_bits(one + 2.0 ** -8) == ref.f64_to_bf16_bits(one)       # tie -> even
    assert ref.f64_to_bf16_bits(one + 3 * 2.0 ** -8) == ref.f64_to_bf16_bits(one + 2.0 ** -6)
    assert ref.f64_to_bf16_bits(one + 2.0 ** -8 + 2.0 ** -30) == ref.f64_to_bf16_bits(one + 2.0 ** -7)
    assert ref.f64_to_bf16_bits(-(one + 2.0 ** -8)) == ref.f64_to_bf16_bits(-one)


def test_position_zero_is_identity():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 128))
    np.testing.assert_array_equal(ref.rope_rotate(x, 0, 500000.0), x)


@pytest.mark.parametrize("pos", [1, 7, 1000, 18431])
def test_two_dims_is_plain_rotation(pos):
    x = np.array([0.3, -1.7])
    got = ref.rope_rotate(x, pos, 10000.0)
    c, s = math.cos(pos), math.sin(pos)
    np.testing.assert_allclose(got, [0.3 * c + 1.7 * s, 0.3 * s - 1.7 * c], rtol=0, atol=1e-12)


def test_pair_norms_preserved():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(64)
    y = ref.rope_rotate(x, 12345, 1e6)
    np.testing.assert_allclose(x[:32] ** 2 + x[32:] ** 2, y[:32] ** 2 + y[32:] ** 2,
                               rtol=1e-12)


def test_dot_products_depend_on_distance_only():
    rng = np.random.default_rng(3)
    a, b = rng.standard_normal(128), rng.standard_normal(128)
    for m, n, d in ((5, 900, 77), (0, 3, 10000), (4000, 100, 1)):
        lhs = ref.rope_rotate(a, m, 500000.0) @ ref.rope_rotate(b, n, 500000.0)
        rhs = ref.rope_rotate(a, m + d, 500000.0) @ ref.rope_rotate(b, n + d, 500000.0)
        assert abs(lhs - rhs) <= 1e-9 * (abs(lhs) + 1)


def test_gather_applies_local_positions():
    rng = np.random.default_rng(4)
    P, H, D = 16, 2, 64
    L = 200
    pages = (L + P - 1) // P
    pt = np.array([rng.permutation(pages)])
    k = ((rng.standard_normal((pages, P, H, D)).astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    v = k.copy()
    scores = rng.random((1, pages * P // 32 + 1))
    kw = dict(page_size=P, chunk_size=32, top_k=2, window=64, capacity=2 * 32 + 64)
    raw = ref.gather_compact(k, v, pt, [L], scores, **kw)
    rot = ref.gather_compact(k, v, pt, [L], scores, rope_base=10000.0, **kw)
    n = int(raw["out_len"][0])
    assert (rot["out_v"] == raw["out_v"]).all()
    assert (rot["out_k"][0, 0] == raw["out_k"][0, 0]).all()      # local position 0
    for i in (1, 5, n - 1):
        want = ref.f64_to_bf16_bits(ref.rope_rotate(ref.bf16_bits_to_f64(raw["out_k"][0, i]), i, 10000.0))
        assert (rot["out_k"][0, i] == want).all()
    assert not (rot["out_k"][0, 1:n] == raw["out_k"][0, 1:n]).all()
