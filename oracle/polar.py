"""PolarQuant variant: recursive polar encoding of rotated K/V vectors, in fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[P3] "PolarQuant: 極座標変換で量子化定数を不要にする": a d-dimensional vector is
turned into polar form recursively.  Its coordinate pairs become d/2 radii and
d/2 angles, the radii are paired and transformed again, and so on until one
radius and d - 1 angles are left.  The angles of (near-)random high-dimensional
vectors have a narrow, known distribution, so every angle is quantized on one
fixed uniform grid and no per-block scale or zero point is stored; the single
radius is kept in fp16 (2 bytes per vector), and the decoder multiplies it back
in (the page's diagram: radius fp16, angles uniformly quantized, combined on
restore).

Readings (the page leaves these open; fixed in include/tq.h):
* The vector is first rotated by the layer's Hadamard rotation Pi (the same
  preconditioning as the TurboQuant layers), which makes the coordinates look
  random so that the angle distribution the page relies on holds.
* Level 1 angle of pair i: atan2(y[2i+1], y[2i]) on the full circle; level
  l >= 2: atan2(rho[2i+1], rho[2i]) of the level below's radii, in [0, pi/2].
* b bits per angle.  Level 1: 2^b equal cells of the circle, starting at
  theta = -pi (code = floor((theta + pi) / (2 pi / 2^b)) mod 2^b, so theta = pi
  and theta = -pi share code 0).  Levels >= 2: 2^b equal cells of [0, pi/2].
  A pair of two zeros has angle 0.  Reconstruction at the cell midpoints.
* Radius r = fp16(||x||), round to nearest even (||x|| = ||Pi x||).
* Record: slot s holds angle code s, levels in order (level 1's d/2 angles,
  then level 2's d/4, ..., the last level's one angle at slot d - 2), slot
  d - 1 = 0, packed as the LSB-first bitstream of the TurboQuant records.
  Page: [16 records of d*b/8 bytes][16 x fp16 radius, little-endian].

Pinned by (tests/test_oracle_polar.py): hand-derived codes of basis vectors
and of 45-degree pairs under Pi = I; each code is the nearest grid midpoint to
the angle computed without the recursion (norms of coordinate blocks);
||direction|| = 1 for any codes; re-encoding a reconstructed vector returns
its codes; ||x_hat|| = r; the direction error stays inside the half-cell bound
summed over levels; higher-level angles concentrate around pi/4 more tightly
level by level (the page's concentration argument); page sizes and the page
round trip.
"""

import numpy as np

from . import pack
from .attention import softmax_weights, token_slots

BLOCK = pack.BLOCK


def num_levels(d):
    n = int(round(np.log2(d)))
    if (1 << n) != d or d < 2:
        raise ValueError("head_dim must be a power of two")
    return n


def level_span(d, level):
    """(first slot, number of angles) of a level (1-based) in the record."""
    count = d >> level
    start = d - (d >> (level - 1))
    return start, count


def polar_angles(y):
    """Recursive polar transform of rows y [n, d].

    Returns (angles, radius): angles[l - 1] is the [n, d / 2^l] array of level-l
    angles, radius the [n] final radius.
    """
    y = np.atleast_2d(np.asarray(y, dtype=np.float64))
    d = y.shape[-1]
    angles = []
    a, b = y[:, 0::2], y[:, 1::2]
    th = np.arctan2(b, a)
    th[(a == 0) & (b == 0)] = 0.0
    angles.append(th)
    rho = np.hypot(a, b)
    for _ in range(2, num_levels(d) + 1):
        a, b = rho[:, 0::2], rho[:, 1::2]
        th = np.arctan2(b, a)
        th[(a == 0) & (b == 0)] = 0.0
        angles.append(th)
        rho = np.hypot(a, b)
    return angles, rho[:, 0]


def cell_width(bits, level):
    """Grid step of a level: the circle (level 1) or [0, pi/2] in 2^bits cells."""
    return (2.0 * np.pi if level == 1 else 0.5 * np.pi) / (1 << bits)


def angle_codes(theta, bits, level):
    """Uniform-grid code of angles of one level."""
    theta = np.asarray(theta, dtype=np.float64)
    n = 1 << bits
    w = cell_width(bits, level)
    if level == 1:
        k = np.floor((theta + np.pi) / w).astype(np.int64)
        return np.mod(k, n)
    k = np.floor(theta / w).astype(np.int64)
    return np.clip(k, 0, n - 1)


def midpoint_angles(codes, bits, level):
    """Reconstruction angle (cell midpoint) of codes of one level."""
    w = cell_width(bits, level)
    mid = (np.asarray(codes, dtype=np.float64) + 0.5) * w
    return mid - np.pi if level == 1 else mid


def radius_fp16(x):
    """r = fp16(||x||) per row, returned as float64."""
    n = np.sqrt(np.sum(np.square(np.atleast_2d(np.asarray(x, dtype=np.float64))), axis=-1))
    return n.astype(np.float16).astype(np.float64)


def encode(x, pi, bits):
    """Rows x [n, d] -> (codes int64 [n, d] in slot order, r float64 [n])."""
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    d = x.shape[-1]
    y = x @ np.asarray(pi, dtype=np.float64).T
    angles, _ = polar_angles(y)
    codes = np.zeros(x.shape, dtype=np.int64)
    for level, th in enumerate(angles, start=1):
        s, c = level_span(d, level)
        codes[:, s:s + c] = angle_codes(th, bits, level)
    return codes, radius_fp16(x)


def direction(codes, bits):
    """Unit direction y_hat [n, d] of rows of slot codes [n, d]."""
    codes = np.atleast_2d(np.asarray(codes, dtype=np.int64))
    n, d = codes.shape
    u = np.ones((n, 1))
    for level in range(num_levels(d), 0, -1):
        s, c = level_span(d, level)
        th = midpoint_angles(codes[:, s:s + c], bits, level)
        child = np.empty((n, 2 * c))
        child[:, 0::2] = u * np.cos(th)
        child[:, 1::2] = u * np.sin(th)
        u = child
    return u


def decode(codes, r, pi, bits):
    """x_hat = r Pi^T y_hat for rows of codes [n, d] and radii r [n]."""
    yh = direction(codes, bits)
    return np.asarray(r, dtype=np.float64)[:, None] * (yh @ np.asarray(pi, dtype=np.float64))


def page_bytes(d, bits):
    return BLOCK * pack.record_bytes(d, bits) + BLOCK * 2


def write_pages(pool, slots, head, num_kv_heads, d, bits, codes, r):
    """Store records and radii of the given slots (slot < 0 skipped) into a flat uint8 pool."""
    pb = page_bytes(d, bits)
    rb = pack.record_bytes(d, bits)
    recs = pack.pack_records(codes, bits)
    rad = np.asarray(r, dtype=np.float64).astype("<f2").view(np.uint8).reshape(-1, 2)
    for i, s in enumerate(np.asarray(slots, dtype=np.int64)):
        if s < 0:
            continue
        blk, off = int(s) // BLOCK, int(s) % BLOCK
        base = (blk * num_kv_heads + head) * pb
        pool[base + off * rb: base + (off + 1) * rb] = recs[i]
        pool[base + BLOCK * rb + 2 * off: base + BLOCK * rb + 2 * off + 2] = rad[i]


def split_pages(pages, d, bits):
    """Pages [..., page_bytes] -> (codes [..., 16, d], r float64 [..., 16])."""
    pages = np.asarray(pages, dtype=np.uint8)
    rb = pack.record_bytes(d, bits)
    lead = pages.shape[:-1]
    codes = pack.unpack_records(pages[..., : BLOCK * rb].reshape(lead + (BLOCK, rb)), bits, d)
    rr = pages[..., BLOCK * rb: BLOCK * rb + 2 * BLOCK].copy()
    r = rr.view("<f2").reshape(lead + (BLOCK,)).astype(np.float64)
    return codes, r


def gather(k_pool, v_pool, pi, bits_k, bits_v, num_blocks, num_kv_heads, d, block_table_row, ctx, head):
    """Decoded keys and values [ctx, d] of one (sequence, kv head) of a polar layer."""
    kp = pack.pool_pages(k_pool, num_blocks, num_kv_heads, page_bytes(d, bits_k))
    vp = pack.pool_pages(v_pool, num_blocks, num_kv_heads, page_bytes(d, bits_v))
    slots = token_slots(block_table_row, ctx)
    blocks, toks = slots // BLOCK, slots % BLOCK
    sel = np.arange(ctx)
    kc, kr = split_pages(kp[blocks, head], d, bits_k)
    vc, vr = split_pages(vp[blocks, head], d, bits_v)
    k_hat = decode(kc[sel, toks], kr[sel, toks], pi, bits_k)
    v_hat = decode(vc[sel, toks], vr[sel, toks], pi, bits_v)
    return k_hat, v_hat


def decode_attention(q, k_pool, v_pool, pi, bits_k, bits_v, num_blocks, num_kv_heads, block_table, context_lens,
                     sm_scale):
    """q [B, H_q, d] -> out [B, H_q, d]: exact softmax attention over the decoded polar cache."""
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    g = hq // num_kv_heads
    out = np.zeros_like(q)
    for b in range(bsz):
        ctx = int(context_lens[b])
        if ctx == 0:
            continue
        for kvh in range(num_kv_heads):
            k_hat, v_hat = gather(k_pool, v_pool, pi, bits_k, bits_v, num_blocks, num_kv_heads, d,
                                  block_table[b], ctx, kvh)
            for h in range(kvh * g, (kvh + 1) * g):
                out[b, h] = softmax_weights(sm_scale * (k_hat @ q[b, h])) @ v_hat
    return out
