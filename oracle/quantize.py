"""Stage-1 quantizer: rotate, normalise, per-coordinate Lloyd-Max code, norm.

[P1] §第1段: rotate the vector, then quantize each coordinate with the
Lloyd-Max scalar quantizer.  [P1] §第2段 (last sentences): vLLM's presets use
stage 1 plus norm correction (`_nc`).  [P2] "Bugs Nobody Else Has Found": the
per-vector norm must be fp32 (fp16 norms broke output at ~11.4K tokens).

Steps, in the order the method applies them (reading fixed in include/tq.h):
  n     = ||x||_2                      (fp64 here, from the input as given)
  y     = Pi x / n                     (unit vector in the rotated domain)
  idx_j = #{ i : y_j >= beta_i }       (ties go to the upper cell)
  gamma = n / ||c[idx]||_2             (norm correction, TQ_NORM_CORRECTED)
        = n                            (TQ_NORM_RAW)
  zero vector: gamma = 0, idx_j = 2^(b-1).
Reconstruction: x_hat = gamma * Pi^T c[idx].

Pinned by (tests/test_oracle_quantize.py): brute-force nearest centroid on
random inputs, constructed exact ties resolve upward, ||x_hat|| = ||x|| for the
corrected norm, zero-vector case, scale equivariance.
"""

import numpy as np

NORM_CORRECTED = 0
NORM_RAW = 1


def bf16_bits_to_f64(u16):
    """Widen bf16 bit patterns (uint16) to float64 exactly."""
    u32 = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def codes_from_y(y, boundaries):
    """idx_j = #{i : y_j >= beta_i}.  Both operands are compared exactly as given."""
    y = np.asarray(y)
    b = np.asarray(boundaries)
    return np.sum(y[..., None] >= b, axis=-1).astype(np.int64)


def quantize(x, pi, centroids, boundaries, norm_mode=NORM_CORRECTED):
    """x: [..., d] float64.  Returns (idx int64 [..., d], gamma f64 [...], y f64 [..., d])."""
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(centroids, dtype=np.float64)
    beta = np.asarray(boundaries, dtype=np.float64)
    d = x.shape[-1]
    n = np.sqrt(np.sum(x * x, axis=-1))
    rot = x @ np.asarray(pi, dtype=np.float64).T          # Pi x for every vector
    safe = np.where(n > 0, n, 1.0)
    y = rot / safe[..., None]
    idx = codes_from_y(y, beta)
    zero = n == 0
    idx[zero] = c.shape[0] // 2
    y[zero] = 0.0
    if norm_mode == NORM_RAW:
        gamma = n.copy()
    else:
        cn = np.sqrt(np.sum(c[idx] ** 2, axis=-1))
        gamma = np.where(zero, 0.0, n / np.where(cn > 0, cn, 1.0))
    del d
    return idx, gamma, y


def dequantize(idx, gamma, pi, centroids):
    """x_hat = gamma * Pi^T c[idx]."""
    c = np.asarray(centroids, dtype=np.float64)
    vals = c[np.asarray(idx)] * np.asarray(gamma, dtype=np.float64)[..., None]
    return vals @ np.asarray(pi, dtype=np.float64)
