"""Stage 2: 1-bit QJL residual for keys.

[P3] "QJL: Johnson-Lindenstrauss変換で残差を1ビット補正する": the stage-1
residual e = x - x_hat is projected by a random matrix R (z = R e) and only the
signs of z are kept (1 bit per dimension, 16 B at d = 128); the query is kept
at high precision and projected by the same R; the score is the stage-1 term
plus a QJL correction whose expectation exactly compensates the quantization
error of the inner product; R is generated once and shared by all layers and
heads.  [P1] §第2段: the purpose is an unbiased inner-product estimate.

Readings (fixed in include/tq.h): the residual is taken in the rotated domain at
full scale, r = Pi x - gamma c[idx] (equal to Pi (x - x_hat)); R = S is m x d
with iid N(0, 1) entries, m = d; sigma_i = [ (S r)_i >= 0 ]; rho = ||r||_2 is
stored as fp32 (the estimator cannot be unbiased without it).  Estimate:

    <q, x>  ~=  gamma <Pi q, c[idx]>
               + sqrt(pi/2) / m * rho * sum_i (2 sigma_i - 1) (S Pi q)_i

which is unbiased over S because E[sign(<s, r>) <s, u>] = sqrt(2/pi) <u, r>/||r||
for s ~ N(0, I).

Pinned by (tests/test_oracle_qjl.py): mean over 10^4 independent S of
(estimate - <q, x>) within 4 standard errors of 0; empirical variance below
pi/(2m) ||Pi q||^2 rho^2; rho = 0 gives a zero correction.
"""

import math

import numpy as np

from .quantize import quantize


def residual_encode(x, pi, centroids, boundaries, s, norm_mode=0):
    """Stage 1 + QJL for key vectors x [n, d].

    Returns (idx [n, d], gamma [n], signs [n, m] in {0,1}, rho [n], r [n, d]).
    """
    x = np.asarray(x, dtype=np.float64)
    idx, gamma, _ = quantize(x, pi, centroids, boundaries, norm_mode)
    r = x @ np.asarray(pi, dtype=np.float64).T - gamma[:, None] * np.asarray(centroids, dtype=np.float64)[idx]
    z = r @ np.asarray(s, dtype=np.float64).T
    signs = (z >= 0).astype(np.int64)
    rho = np.sqrt(np.sum(r * r, axis=-1))
    return idx, gamma, signs, rho, r


def estimate(q, pi, centroids, idx, gamma, signs, rho, s):
    """Unbiased estimate of <q, x_t> for every token t.  q [d]; idx [T, d]; returns [T]."""
    q = np.asarray(q, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    m = s.shape[0]
    qr = np.asarray(pi, dtype=np.float64) @ q
    u = s @ qr
    c = np.asarray(centroids, dtype=np.float64)
    stage1 = np.asarray(gamma, dtype=np.float64) * (c[np.asarray(idx)] @ qr)
    pm = 2.0 * np.asarray(signs, dtype=np.float64) - 1.0
    corr = math.sqrt(math.pi / 2.0) / m * np.asarray(rho, dtype=np.float64) * (pm @ u)
    return stage1 + corr
