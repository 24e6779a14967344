"""Seeded random draws used by the method itself (rotation signs, Gaussian
matrices for the dense rotation and the QJL projection).

The pages fix no generator ([P1] §第1段 only says "random rotation"; [P3]'s QJL
section says the projection R is generated once at start-up and shared by all
layers and heads).  The reading fixed in ``include/tq.h`` is Vigna's
SplitMix64, implemented here from its published definition:

    state += 0x9E3779B97F4A7C15
    z = state
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB
    return z ^ (z >> 31)            (all arithmetic mod 2**64)

Stream key: state0 = seed XOR ((kind * 2**32 + layer) * 0x9E3779B97F4A7C15).

* sign i      : -1 if bit 63 of draw i is set, else +1
* uniform     : (draw >> 11) * 2**-53  in [0, 1)
* Gaussians   : Box-Muller on consecutive uniform pairs (u1, u2):
                r = sqrt(-2 ln(1 - u1)), g0 = r cos(2 pi u2), g1 = r sin(2 pi u2)
                (g0 first, then g1), filling matrices row-major.

Pinned by: SplitMix64 known-answer values for seed 0, sign balance and Gaussian
moment checks (tests/test_oracle_rng.py).
"""

import math

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15

KIND_HADAMARD = 1
KIND_DENSE = 2
KIND_QJL = 3


def stream_state(seed, kind, layer):
    """Initial SplitMix64 state for a (seed, kind, layer) stream."""
    return (int(seed) ^ (((int(kind) << 32) + int(layer)) * GOLDEN)) & MASK64


def splitmix64(state0, n):
    """n successive SplitMix64 outputs from state0 (Python ints)."""
    out = []
    s = state0 & MASK64
    for _ in range(n):
        s = (s + GOLDEN) & MASK64
        z = s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        out.append(z ^ (z >> 31))
    return out


def signs(seed, layer, n, kind=KIND_HADAMARD):
    """+-1 vector (float64) from the top bit of each draw."""
    draws = splitmix64(stream_state(seed, kind, layer), n)
    return np.array([-1.0 if (z >> 63) else 1.0 for z in draws], dtype=np.float64)


def uniforms(state0, n):
    draws = splitmix64(state0, n)
    return np.array([(z >> 11) * 2.0 ** -53 for z in draws], dtype=np.float64)


def gaussians(seed, kind, layer, n):
    """n standard normals by Box-Muller (cos branch, then sin branch)."""
    npairs = (n + 1) // 2
    u = uniforms(stream_state(seed, kind, layer), 2 * npairs)
    out = np.empty(2 * npairs, dtype=np.float64)
    for p in range(npairs):
        u1 = 1.0 - u[2 * p]
        u2 = u[2 * p + 1]
        r = math.sqrt(-2.0 * math.log(u1))
        out[2 * p] = r * math.cos(2.0 * math.pi * u2)
        out[2 * p + 1] = r * math.sin(2.0 * math.pi * u2)
    return out[:n]


def gaussian_matrix(seed, kind, layer, rows, cols):
    return gaussians(seed, kind, layer, rows * cols).reshape(rows, cols)
