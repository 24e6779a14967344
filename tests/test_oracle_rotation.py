"""Pins for the oracle's rotations (CPU only)."""
import numpy as np
import pytest

from oracle import rng, rotation


@pytest.mark.parametrize("d", [1, 2, 4, 16, 128, 256])
def test_sylvester_closed_form(d):
    h = rotation.sylvester_hadamard(d)
    i = np.arange(d)
    pop = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    assert np.array_equal(h, (-1.0) ** pop)


def fwht_butterfly(x):
    """Textbook in-place fast Walsh-Hadamard butterfly (unnormalised)."""
    x = np.array(x, dtype=np.float64)
    h = 1
    while h < x.shape[0]:
        for i in range(0, x.shape[0], 2 * h):
            a = x[i:i + h].copy()
            b = x[i + h:i + 2 * h].copy()
            x[i:i + h] = a + b
            x[i + h:i + 2 * h] = a - b
        h *= 2
    return x


def test_fwht_equals_matrix():
    g = np.random.default_rng(1)
    for d in (2, 8, 64, 128):
        x = g.standard_normal(d)
        assert np.allclose(fwht_butterfly(x), rotation.sylvester_hadamard(d) @ x, atol=1e-12)


def test_hadamard_rotation_orthogonal_and_seeded():
    d = 128
    pi = rotation.hadamard_rotation_seeded(0, 0, d)
    assert np.max(np.abs(pi @ pi.T - np.eye(d))) < 1e-13
    x = np.random.default_rng(2).standard_normal(d)
    assert abs(np.linalg.norm(pi @ x) - np.linalg.norm(x)) < 1e-12
    s = rng.signs(0, 0, d)
    # Pi e_j = s_j H[:, j] / sqrt(d): first row of Pi is s / sqrt(d)
    assert np.allclose(pi[0], s / np.sqrt(d), atol=1e-15)
    # H_d e_0 = 1/sqrt(d) (all ones column) up to the sign s_0
    assert np.allclose(pi[:, 0] * s[0], np.ones(d) / np.sqrt(d), atol=1e-15)


def gram_schmidt(g):
    """Modified Gram-Schmidt on the columns of g: Q with positive diag(R)."""
    g = np.array(g, dtype=np.float64)
    n = g.shape[1]
    q = np.zeros_like(g)
    for j in range(n):
        v = g[:, j].copy()
        for _ in range(2):  # re-orthogonalise once for fp64 accuracy
            for i in range(j):
                v -= (q[:, i] @ v) * q[:, i]
        q[:, j] = v / np.linalg.norm(v)
    return q


def test_dense_rotation_is_unique_haar_q():
    d = 128
    pi = rotation.dense_rotation_seeded(7, 3, d)
    assert np.max(np.abs(pi @ pi.T - np.eye(d))) < 1e-13
    g = rng.gaussian_matrix(7, rng.KIND_DENSE, 3, d, d)
    # QR with positive diag(R) is unique: an independent Gram-Schmidt agrees
    assert np.max(np.abs(gram_schmidt(g) - pi)) < 1e-10
    # R = Pi^T G is upper triangular with positive diagonal
    r = pi.T @ g
    assert np.max(np.abs(np.tril(r, -1))) < 1e-10
    assert np.all(np.diag(r) > 0)


def test_layers_and_kinds_differ():
    a = rotation.dense_rotation_seeded(0, 0, 16)
    b = rotation.dense_rotation_seeded(0, 1, 16)
    assert np.max(np.abs(a - b)) > 0.1
    s = rotation.qjl_matrix_seeded(0, 128, 128)
    assert s.shape == (128, 128)
    assert abs(s.mean()) < 4 / 128 and abs(s.var() - 1) < 0.05
