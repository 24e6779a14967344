"""Lloyd-Max codebook for one coordinate of a randomly rotated unit vector.

[P1] §第1段: after the random rotation each coordinate gets a Lloyd-Max scalar
quantizer (representatives placed optimally for the value distribution); [P1]
§キャリブレーション: no calibration data is used, so the distribution is fixed
in advance.

Reading (the pages give no formula): after a Haar rotation the coordinate t of
a unit vector in R^d has density

    f_d(t) = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)) * (1 - t^2)^((d-3)/2),  |t| <= 1

(t^2 ~ Beta(1/2, (d-1)/2)).  The quantizer with 2^b cells is found by Lloyd's
iteration in fp64:

    beta_i = (c_i + c_{i+1}) / 2                       (midpoint condition)
    c_i    = E[t | beta_{i-1} <= t < beta_i]           (centroid condition)

with beta_{-1} = -1, beta_{2^b - 1} = +1, started from the quantiles
F^{-1}((i + 1/2) / 2^b) and stopped when max |delta c| < 1e-15.  The cell mass
uses the regularised incomplete beta function; the cell first moment has the
closed form  int_a^b t f(t) dt = K/(d-1) [(1-a^2)^((d-1)/2) - (1-b^2)^((d-1)/2)].

Emission (what the kernels use): c32 = fp32(c) for the upper half, mirrored
(c32[2^b-1-i] = -c32[i]) so the table is exactly antisymmetric;
beta32_i = fp32(fp32(c32_i + c32_{i+1}) * 0.5), i.e. the fp32 midpoint of the
fp32 centroids computed in fp32.

Pinned by (tests/test_oracle_codebook.py): normalisation and E[t^2] = 1/d of
the density; centroid condition re-checked with scipy.integrate.quad on the
density itself; b = 1 closed form c = +-Gamma(d/2)/(sqrt(pi) Gamma((d+1)/2));
large-d limit against the Gaussian Lloyd-Max quantizer (Max, 1960);
distortion strictly decreasing in b; symmetry.
"""

import math

import numpy as np
from scipy import special


def density_const(d):
    return math.exp(math.lgamma(d / 2.0) - math.lgamma((d - 1) / 2.0)) / math.sqrt(math.pi)


def density(t, d):
    t = np.asarray(t, dtype=np.float64)
    return density_const(d) * np.power(np.clip(1.0 - t * t, 0.0, None), (d - 3) / 2.0)


def _upper_tail(t, d):
    """P(T >= t) for t >= 0, without cancellation."""
    return 0.5 * special.betaincc(0.5, (d - 1) / 2.0, t * t)


def cdf(t, d):
    t = float(t)
    if t >= 1.0:
        return 1.0
    if t <= -1.0:
        return 0.0
    if t >= 0.0:
        return 1.0 - _upper_tail(t, d)
    return _upper_tail(-t, d)


def cell_mass(a, b, d):
    """P(a <= T < b) computed without catastrophic cancellation."""
    a = max(float(a), -1.0)
    b = min(float(b), 1.0)
    if b <= a:
        return 0.0
    if a >= 0.0:
        return _upper_tail(a, d) - _upper_tail(b, d)
    if b <= 0.0:
        return _upper_tail(-b, d) - _upper_tail(-a, d)
    return 1.0 - _upper_tail(-a, d) - _upper_tail(b, d)


def cell_moment(a, b, d):
    """int_a^b t f_d(t) dt (closed form)."""
    a = max(float(a), -1.0)
    b = min(float(b), 1.0)
    e = (d - 1) / 2.0
    return density_const(d) / (d - 1) * ((1.0 - a * a) ** e - (1.0 - b * b) ** e)


def quantile(p, d):
    """F^{-1}(p) via the inverse regularised incomplete beta."""
    if p == 0.5:
        return 0.0
    if p > 0.5:
        return math.sqrt(special.betaincinv(0.5, (d - 1) / 2.0, 2.0 * p - 1.0))
    return -quantile(1.0 - p, d)


def lloyd_max(d, bits, tol=1e-15, max_iter=200000):
    """fp64 Lloyd iteration.  Returns (centroids[2^b], boundaries[2^b - 1], iters)."""
    k = 1 << bits
    c = np.array([quantile((i + 0.5) / k, d) for i in range(k)], dtype=np.float64)
    for it in range(1, max_iter + 1):
        beta = 0.5 * (c[:-1] + c[1:])
        edges = np.concatenate(([-1.0], beta, [1.0]))
        new = np.array([cell_moment(edges[i], edges[i + 1], d) / cell_mass(edges[i], edges[i + 1], d)
                        for i in range(k)])
        delta = np.max(np.abs(new - c))
        c = new
        if delta < tol:
            return c, 0.5 * (c[:-1] + c[1:]), it
    raise RuntimeError("Lloyd iteration did not converge")


def emit_fp32(c):
    """fp32 tables the kernels consume (see module docstring)."""
    c = np.asarray(c, dtype=np.float64)
    k = c.shape[0]
    half = k // 2
    c32 = np.empty(k, dtype=np.float32)
    c32[half:] = c[half:].astype(np.float32)
    c32[:half] = -c32[half:][::-1]
    b32 = ((c32[:-1] + c32[1:]).astype(np.float32) * np.float32(0.5)).astype(np.float32)
    return c32, b32


_CACHE = {}


def codebook_fp32(d, bits):
    key = (d, bits)
    if key not in _CACHE:
        c, _, _ = lloyd_max(d, bits)
        _CACHE[key] = emit_fp32(c)
    return _CACHE[key]


def distortion(c, beta, d):
    """E[(T - Q(T))^2] for the quantizer (c, beta) under f_d (fp64 quadrature)."""
    from scipy import integrate
    edges = np.concatenate(([-1.0], np.asarray(beta, dtype=np.float64), [1.0]))
    total = 0.0
    for i, ci in enumerate(c):
        val, _ = integrate.quad(lambda t: (t - ci) ** 2 * float(density(t, d)),
                                edges[i], edges[i + 1], epsabs=1e-16, epsrel=1e-12, limit=200)
        total += val
    return total
