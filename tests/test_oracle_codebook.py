"""Pins for the oracle's Lloyd-Max codebook (CPU only)."""
import math

import numpy as np
import pytest
from scipy import integrate

from oracle import codebook as cb

# Gaussian Lloyd-Max quantizer (J. Max, "Quantizing for minimum distortion",
# IRE Trans. Inf. Theory, 1960): positive output levels and MSE for unit variance.
MAX1960_LEVELS = {
    1: [0.7979],
    2: [0.4528, 1.510],
    3: [0.2451, 0.7560, 1.344, 2.152],
    4: [0.1284, 0.3881, 0.6568, 0.9424, 1.256, 1.618, 2.069, 2.733],
}
MAX1960_MSE = {1: 0.3634, 2: 0.1175, 3: 0.03454, 4: 0.009497}


@pytest.mark.parametrize("d", [16, 128, 256])
def test_density_normalised_and_variance(d):
    one, _ = integrate.quad(lambda t: float(cb.density(t, d)), -1, 1, epsabs=1e-14, limit=200)
    var, _ = integrate.quad(lambda t: t * t * float(cb.density(t, d)), -1, 1, epsabs=1e-14, limit=200)
    assert abs(one - 1.0) < 1e-10
    # coordinate of a uniform unit vector: E[t^2] = 1/d
    assert abs(var - 1.0 / d) < 1e-12


def test_closed_forms_against_quadrature():
    d = 128
    for a, b in [(-1.0, -0.2), (-0.05, 0.03), (0.0, 0.1), (0.1, 0.25), (0.3, 1.0)]:
        mass, _ = integrate.quad(lambda t: float(cb.density(t, d)), a, b, epsabs=1e-16, epsrel=1e-12)
        mom, _ = integrate.quad(lambda t: t * float(cb.density(t, d)), a, b, epsabs=1e-16, epsrel=1e-12)
        assert abs(cb.cell_mass(a, b, d) - mass) < 1e-12 + 1e-9 * mass
        assert abs(cb.cell_moment(a, b, d) - mom) < 1e-13 + 1e-9 * abs(mom)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_lloyd_fixed_point_conditions(bits):
    d = 128
    c, beta, _ = cb.lloyd_max(d, bits)
    k = 1 << bits
    assert np.all(np.diff(c) > 0)
    # symmetry of the optimum for a symmetric density
    assert np.max(np.abs(c + c[::-1])) < 1e-13
    assert abs(beta[k // 2 - 1]) < 1e-14
    # midpoint condition
    assert np.max(np.abs(beta - 0.5 * (c[:-1] + c[1:]))) < 1e-15
    # centroid condition, re-checked with direct quadrature of the density
    edges = np.concatenate(([-1.0], beta, [1.0]))
    for i in range(k):
        num, _ = integrate.quad(lambda t: t * float(cb.density(t, d)), edges[i], edges[i + 1],
                                epsabs=1e-17, epsrel=1e-13, limit=200)
        den, _ = integrate.quad(lambda t: float(cb.density(t, d)), edges[i], edges[i + 1],
                                epsabs=1e-17, epsrel=1e-13, limit=200)
        assert abs(num / den - c[i]) < 1e-11


@pytest.mark.parametrize("d", [8, 128, 1000])
def test_one_bit_closed_form(d):
    c, _, _ = cb.lloyd_max(d, 1)
    e_abs = math.exp(math.lgamma(d / 2) - math.lgamma((d + 1) / 2)) / math.sqrt(math.pi)
    assert abs(c[1] - e_abs) < 1e-13 and abs(c[0] + e_abs) < 1e-13
    if d == 128:
        assert abs(math.sqrt(d) * c[1] - 0.79944) < 5e-6


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_large_d_limit_is_gaussian_lloyd_max(bits):
    d = 1 << 16
    # at this d the fp64 cell moments carry ~1e-14 noise, so stop earlier
    c, beta, _ = cb.lloyd_max(d, bits, tol=1e-12)
    levels = math.sqrt(d) * c[len(c) // 2:]
    assert np.max(np.abs(levels - np.array(MAX1960_LEVELS[bits]))) < 1.5e-3
    mse = d * cb.distortion(c, beta, d)
    assert abs(mse - MAX1960_MSE[bits]) < 2e-3 * MAX1960_MSE[bits] + 5e-5
    # and the finite-d levels move toward the limit as d grows
    c_small, _, _ = cb.lloyd_max(64, bits)
    small = 8.0 * c_small[len(c_small) // 2:]
    assert np.max(np.abs(small - MAX1960_LEVELS[bits])) > np.max(np.abs(levels - MAX1960_LEVELS[bits]))


def test_distortion_decreases_with_bits():
    d = 128
    dist = []
    for bits in (1, 2, 3, 4):
        c, beta, _ = cb.lloyd_max(d, bits)
        dist.append(cb.distortion(c, beta, d))
    assert all(a > b for a, b in zip(dist, dist[1:]))
    # every Lloyd-Max quantizer beats the trivial one (E[t^2] = 1/d)
    assert dist[0] < 1.0 / d


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_emitted_tables(bits):
    c32, b32 = cb.codebook_fp32(128, bits)
    assert c32.dtype == np.float32 and b32.dtype == np.float32
    assert np.array_equal(c32, -c32[::-1])
    assert np.all(np.diff(c32) > 0) and np.all(np.diff(b32) > 0)
    assert b32[len(b32) // 2] == 0.0
    mid = ((c32[:-1] + c32[1:]).astype(np.float32) * np.float32(0.5))
    assert np.array_equal(mid, b32)
    c, _, _ = cb.lloyd_max(128, bits)
    assert np.max(np.abs(c32.astype(np.float64) - c)) < 1e-8
