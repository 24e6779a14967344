"""Pins for the oracle's QJL residual estimator (CPU only)."""
import math

import numpy as np

from oracle import codebook as cb, qjl, rotation


def test_estimator_unbiased_over_projections():
    d, bits, trials = 128, 2, 10000
    c32, b32 = cb.codebook_fp32(d, bits)
    pi = rotation.hadamard_rotation_seeded(0, 0, d)
    g = np.random.default_rng(10)
    x = g.standard_normal((1, d))
    q = g.standard_normal(d)
    truth = float(q @ x[0])
    est = np.empty(trials)
    for i in range(trials):
        s = g.standard_normal((d, d))
        idx, gamma, signs, rho, _ = qjl.residual_encode(x, pi, c32, b32, s)
        est[i] = qjl.estimate(q, pi, c32, idx, gamma, signs, rho, s)[0]
    se = est.std(ddof=1) / math.sqrt(trials)
    assert abs(est.mean() - truth) < 4 * se
    # stage 1 alone is biased for this (q, x): the correction is doing the work
    idx, gamma, _, rho, r = qjl.residual_encode(x, pi, c32, b32, np.eye(d))
    stage1 = gamma[0] * (c32[idx[0]] @ (pi @ q))
    assert abs(stage1 - truth) > 8 * se
    # variance of sign-JL estimate is at most pi/(2m) ||Pi q||^2 rho^2
    bound = math.pi / (2 * d) * float(np.sum((pi @ q) ** 2)) * rho[0] ** 2
    assert est.var(ddof=1) <= bound * 1.05


def test_zero_residual_gives_zero_correction():
    d = 128
    c32, _ = cb.codebook_fp32(d, 2)
    pi = np.eye(d)
    idx = np.random.default_rng(1).integers(0, 4, size=(3, d))
    gamma = np.array([1.0, 2.0, 0.5])
    signs = np.random.default_rng(2).integers(0, 2, size=(3, d))
    q = np.random.default_rng(3).standard_normal(d)
    s = np.random.default_rng(4).standard_normal((d, d))
    est = qjl.estimate(q, pi, c32, idx, gamma, signs, np.zeros(3), s)
    assert np.allclose(est, gamma * (c32[idx] @ q), atol=1e-14)


def test_residual_is_rotated_quantization_error():
    d = 128
    c32, b32 = cb.codebook_fp32(d, 2)
    pi = rotation.hadamard_rotation_seeded(3, 1, d)
    x = np.random.default_rng(5).standard_normal((4, d))
    s = np.random.default_rng(6).standard_normal((d, d))
    idx, gamma, signs, rho, r = qjl.residual_encode(x, pi, c32, b32, s)
    xhat = (c32[idx] * gamma[:, None]) @ pi
    assert np.allclose(r, (x - xhat) @ pi.T, atol=1e-12)
    assert np.allclose(rho, np.linalg.norm(x - xhat, axis=1), atol=1e-12)
    assert np.array_equal(signs, ((r @ s.T) >= 0).astype(np.int64))
