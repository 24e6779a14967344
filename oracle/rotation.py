"""Per-layer rotations and the QJL projection, as explicit fp64 matrices.

[P1] §第1段: every K/V vector is multiplied by a random rotation before the
per-coordinate scalar quantizer, which evens out outlier channels.
[P1] §llama.cpp本家: the Hadamard form (fast Walsh-Hadamard transform of Q/K/V
before the cache) is what llama.cpp adopted.

Readings (fixed in include/tq.h):
* Hadamard kind: Pi = H_d diag(s) / sqrt(d), H_d the Sylvester Hadamard matrix
  (H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]), s the +-1 sign stream of
  (seed, kind=1, layer).  One sign layer, one H.
* Dense kind: G = d x d Gaussian from the (seed, kind=2, layer) stream,
  row-major; G = Q R (any QR); Pi = Q diag(sign(diag R)).  This Q is unique, so
  every correct QR gives the same Pi (Haar-distributed).
* QJL projection S: m x d Gaussian (m = d) from (seed, kind=3, layer=0); the
  same S serves every layer and head ([P3] QJL section).
* One rotation per layer, shared by K, V and all heads of the layer.

The oracle applies rotations as plain matrix products (no fast transform).
Pinned by: Sylvester closed form H[i, j] = (-1)^popcount(i & j), orthogonality,
norm preservation, QR uniqueness (tests/test_oracle_rotation.py).
"""

import numpy as np

from . import rng


def sylvester_hadamard(d):
    """Sylvester recursion H_{2n} = [[H_n, H_n], [H_n, -H_n]]."""
    if d < 1 or (d & (d - 1)) != 0:
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1), dtype=np.float64)
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def hadamard_rotation(signs):
    """Pi = H_d diag(signs) / sqrt(d)."""
    signs = np.asarray(signs, dtype=np.float64)
    d = signs.shape[0]
    return sylvester_hadamard(d) * signs[None, :] / np.sqrt(d)


def hadamard_rotation_seeded(seed, layer, d):
    return hadamard_rotation(rng.signs(seed, layer, d, kind=rng.KIND_HADAMARD))


def haar_from_gaussian(g):
    """Pi = Q diag(sign(diag R)) for G = Q R."""
    q, r = np.linalg.qr(np.asarray(g, dtype=np.float64))
    s = np.sign(np.diag(r))
    s[s == 0] = 1.0
    return q * s[None, :]


def dense_rotation_seeded(seed, layer, d):
    return haar_from_gaussian(rng.gaussian_matrix(seed, rng.KIND_DENSE, layer, d, d))


def qjl_matrix_seeded(seed, m, d):
    return rng.gaussian_matrix(seed, rng.KIND_QJL, 0, m, d)


def rotation_seeded(kind, seed, layer, d):
    if kind == rng.KIND_HADAMARD:
        return hadamard_rotation_seeded(seed, layer, d)
    if kind == rng.KIND_DENSE:
        return dense_rotation_seeded(seed, layer, d)
    raise ValueError("unknown rotation kind")
