"""Pins for the oracle's stage-1 quantizer (CPU only)."""
import numpy as np
import pytest

from oracle import codebook as cb, quantize as oq, rotation


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_boundary_count_equals_brute_force_nearest(bits):
    c32, b32 = cb.codebook_fp32(128, bits)
    g = np.random.default_rng(bits)
    y = (g.standard_normal(200000) / np.sqrt(128)).astype(np.float32)
    # keep values away from the fp32-rounded midpoints
    far = np.min(np.abs(y[:, None].astype(np.float64) - b32[None, :]), axis=1) > 1e-6
    y = y[far]
    idx = oq.codes_from_y(y, b32)
    brute = np.argmin(np.abs(y[:, None].astype(np.float64) - c32[None, :].astype(np.float64)), axis=1)
    assert np.array_equal(idx, brute)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_exact_ties_go_up(bits):
    _, b32 = cb.codebook_fp32(128, bits)
    idx = oq.codes_from_y(b32, b32)
    assert np.array_equal(idx, np.arange(1, len(b32) + 1))
    below = np.nextafter(b32, np.float32(-np.inf))
    assert np.array_equal(oq.codes_from_y(below, b32), np.arange(0, len(b32)))
    # -0.0 compares equal to the middle boundary 0.0 and goes up as well
    assert oq.codes_from_y(np.array([-0.0], np.float32), b32)[0] == len(b32) // 2 + 1


def test_norm_correction_preserves_norm_and_zero_vector():
    d, bits = 128, 4
    c32, b32 = cb.codebook_fp32(d, bits)
    pi = rotation.hadamard_rotation_seeded(0, 0, d)
    g = np.random.default_rng(5)
    x = g.standard_normal((64, d)) * 3.0
    x[7] = 0.0
    idx, gamma, y = oq.quantize(x, pi, c32, b32)
    xh = oq.dequantize(idx, gamma, pi, c32)
    n = np.linalg.norm(x, axis=1)
    assert np.allclose(np.linalg.norm(xh, axis=1), n, rtol=1e-13, atol=0)
    assert gamma[7] == 0.0 and np.all(idx[7] == 8)
    assert np.allclose(np.linalg.norm(y[np.arange(64) != 7], axis=1), 1.0, atol=1e-13)
    # raw norm mode keeps gamma = ||x||
    _, graw, _ = oq.quantize(x, pi, c32, b32, norm_mode=oq.NORM_RAW)
    assert np.allclose(graw, n)


def test_scale_equivariance_and_quality():
    d, bits = 128, 4
    c32, b32 = cb.codebook_fp32(d, bits)
    pi = rotation.hadamard_rotation_seeded(1, 2, d)
    x = np.random.default_rng(6).standard_normal((32, d))
    i1, g1, _ = oq.quantize(x, pi, c32, b32)
    i2, g2, _ = oq.quantize(4.0 * x, pi, c32, b32)
    assert np.array_equal(i1, i2) and np.allclose(g2, 4.0 * g1, rtol=1e-15)
    # 4-bit quantization of Gaussian vectors: relative MSE near d * D_4 ~ 0.0095
    xh = oq.dequantize(i1, g1, pi, c32)
    rel = np.sum((x - xh) ** 2) / np.sum(x ** 2)
    assert 0.004 < rel < 0.02


def test_bf16_widening():
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8000], dtype=np.uint16)
    vals = oq.bf16_bits_to_f64(bits)
    assert vals[0] == 1.0 and vals[1] == -2.0 and vals[2] == 2.0 ** -133
    assert vals[3] == (2 - 2 ** -7) * 2.0 ** 127 and vals[4] == 0.0 and np.signbit(vals[4])
