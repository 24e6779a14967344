"""Pins for the oracle's SplitMix64 streams (CPU only)."""
import math

import numpy as np

from oracle import rng


def test_splitmix64_known_answers():
    # Vigna's public-domain splitmix64.c, first three outputs for state 0.
    out = rng.splitmix64(0, 3)
    assert out == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_stream_key_definition():
    # state0 = seed ^ ((kind << 32) + layer) * golden, mod 2^64
    s = rng.stream_state(5, 2, 7)
    assert s == (5 ^ (((2 << 32) + 7) * 0x9E3779B97F4A7C15)) & ((1 << 64) - 1)
    assert rng.stream_state(0, 1, 0) != rng.stream_state(0, 1, 1)
    assert rng.stream_state(0, 1, 0) != rng.stream_state(0, 2, 0)


def test_signs_balanced_and_deterministic():
    s = rng.signs(0, 0, 20000)
    assert set(np.unique(s)) == {-1.0, 1.0}
    assert abs(s.mean()) < 4.0 / math.sqrt(s.size)
    assert np.array_equal(s, rng.signs(0, 0, 20000))
    assert not np.array_equal(s[:128], rng.signs(0, 1, 128))


def test_uniform_range_and_top_bits():
    draws = rng.splitmix64(rng.stream_state(3, 2, 0), 1000)
    u = rng.uniforms(rng.stream_state(3, 2, 0), 1000)
    assert np.all(u >= 0) and np.all(u < 1)
    assert all(abs(ui - (z >> 11) / 2.0 ** 53) == 0 for ui, z in zip(u, draws))


def test_gaussian_moments():
    g = rng.gaussians(11, rng.KIND_DENSE, 0, 40000)
    n = g.size
    assert abs(g.mean()) < 4 / math.sqrt(n)
    assert abs(g.var() - 1.0) < 4 * math.sqrt(2.0 / n)
    assert abs(np.mean(g ** 4) - 3.0) < 4 * math.sqrt(96.0 / n)
    # Box-Muller pair: g0 = r cos, g1 = r sin -> g0^2 + g1^2 = -2 ln(1 - u1)
    u = rng.uniforms(rng.stream_state(11, rng.KIND_DENSE, 0), 2)
    assert abs(g[0] ** 2 + g[1] ** 2 + 2 * math.log(1 - u[0])) < 1e-12
    assert abs(math.atan2(g[1], g[0]) % (2 * math.pi) - 2 * math.pi * u[1]) < 1e-12
