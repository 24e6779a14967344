"""Pins of the PolarQuant-variant oracle (oracle/polar.py) against what the
definitions and the mathematics fix: hand-derived codes, nearest-midpoint
codes from angles computed without the recursion, unit directions, exact
radius, the half-cell error bound, the page's concentration argument and the
page layout."""
import numpy as np
import pytest

from oracle import pack, polar, rotation as orot

D = 128
EYE = np.eye(D)


def basis(i, scale=1.0):
    x = np.zeros(D)
    x[i] = scale
    return x


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_hand_derived_codes_of_basis_vectors(bits):
    n = 1 << bits
    half, quarter = n // 2, n // 4
    # e0: pair 0 = (1, 0), theta 0 -> phi = pi -> code n/2; all other pairs are zero pairs
    # (theta 0, code n/2); every higher pair is (rho, 0) or (0, 0): theta 0, code 0
    codes, r = polar.encode(basis(0, 3.0), EYE, bits)
    want = np.zeros(D, np.int64)
    want[:64] = half
    assert np.array_equal(codes[0], want) and r[0] == 3.0
    # e1: pair 0 = (0, 1), theta pi/2 -> phi = 3 pi / 2 -> code 3n/4
    codes, _ = polar.encode(basis(1), EYE, bits)
    want1 = want.copy()
    want1[0] = 3 * quarter
    assert np.array_equal(codes[0], want1)
    # e2: level 1 all n/2; level-2 pair 0 = (rho_0, rho_1) = (0, 1): theta pi/2 -> last cell
    codes, _ = polar.encode(basis(2), EYE, bits)
    want2 = want.copy()
    want2[64] = n - 1
    assert np.array_equal(codes[0], want2)
    # e64: level-7 pair = (0, 1) -> slot 126 = n - 1; its level-6 node is the left child
    # of the right half (slot 125 = 0), level 1 pair 32 = (1, 0) -> n/2
    codes, _ = polar.encode(basis(64), EYE, bits)
    want64 = want.copy()
    want64[126] = n - 1
    assert np.array_equal(codes[0], want64)
    # -e0: theta = +-pi -> phi = 2 pi or 0 -> code 0 either way
    codes, _ = polar.encode(basis(0, -1.0), EYE, bits)
    assert codes[0, 0] == 0


def test_hand_derived_codes_of_diagonal_pairs():
    # 4 bits: (1, 1): theta pi/4 -> phi 5 pi / 4 -> floor(10) = 10; (-1, 1): theta 3 pi/4 ->
    # phi 7 pi / 4 -> 14; (1, -1): -pi/4 -> 3 pi / 4 -> 6; (-1, -1): -3 pi/4 -> pi/4 -> 2
    x = np.zeros(D)
    x[0:8] = [1, 1, -1, 1, 1, -1, -1, -1]
    codes, _ = polar.encode(x, EYE, 4)
    assert list(codes[0, :4]) == [10, 14, 6, 2]
    # level 2 over equal radii sqrt(2), sqrt(2): theta pi/4 = 4 cells of pi/32 -> 8 (4 bits)
    assert codes[0, 64] == 8 and codes[0, 65] == 8
    # level 3 pair (2, 2): 8 as well; level 4 pair (|x[0:8]| = 2 sqrt 2, 0) -> 0
    assert codes[0, 96] == 8 and codes[0, 112] == 0


def direct_angles(y, level):
    """Level-l angles without the recursion: norms of coordinate blocks of 2^(l-1)."""
    w = 1 << (level - 1)
    blocks = y.reshape(y.shape[0], -1, w)
    if level == 1:
        a, b = y[:, 0::2], y[:, 1::2]
        return np.arctan2(b, a)
    nrm = np.sqrt(np.sum(blocks ** 2, axis=-1))
    return np.arctan2(nrm[:, 1::2], nrm[:, 0::2])


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codes_are_nearest_midpoints(bits):
    rng = np.random.default_rng(11 + bits)
    x = rng.standard_normal((64, D)) * rng.lognormal(size=(1, D))
    pi = orot.rotation_seeded(1, 5, 2, D)
    codes, _ = polar.encode(x, pi, bits)
    y = x @ pi.T
    n = 1 << bits
    for level in range(1, 8):
        th = direct_angles(y, level)
        s, c = polar.level_span(D, level)
        if level == 1:
            mids = (np.arange(n) + 0.5) * (2 * np.pi / n) - np.pi
            diff = np.abs(th[..., None] - mids)
            dist = np.minimum(diff, 2 * np.pi - diff)  # on the circle
        else:
            mids = (np.arange(n) + 0.5) * (np.pi / 2 / n)
            dist = np.abs(th[..., None] - mids)
        assert np.array_equal(np.argmin(dist, axis=-1), codes[:, s:s + c])
    assert np.all(codes[:, D - 1] == 0)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_direction_is_unit_and_reencodes(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, size=(50, D))
    codes[:, D - 1] = 0
    yh = polar.direction(codes, bits)
    assert np.allclose(np.linalg.norm(yh, axis=1), 1.0, atol=1e-14)
    pi = orot.rotation_seeded(1, 9, 0, D)
    xh = polar.decode(codes, np.full(50, 2.5), pi, bits)
    assert np.allclose(np.linalg.norm(xh, axis=1), 2.5, atol=1e-13)
    back, r = polar.encode(xh, pi, bits)  # midpoints lie inside their cells
    assert np.array_equal(back, codes) and np.all(r == 2.5)


def test_radius_is_fp16_of_the_norm():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((200, D)) * 7.0
    _, r = polar.encode(x, EYE, 4)
    n = np.linalg.norm(x, axis=1)
    assert np.all(np.abs(r - n) <= n * 2.0 ** -11)  # half an fp16 ulp
    assert np.array_equal(r, n.astype(np.float16).astype(np.float64))
    codes, r0 = polar.encode(np.zeros((1, D)), EYE, 3)
    assert r0[0] == 0.0 and np.all(codes[0, :64] == 4) and np.all(codes[0, 64:] == 0)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_direction_error_within_half_cell_bound(bits):
    # moving every angle of one level by at most delta moves the unit direction by at
    # most delta (the level's nodes split the unit vector into orthogonal parts);
    # summed over levels: pi / 2^b (level 1) + 6 * pi / 2^(b+2)
    rng = np.random.default_rng(20 + bits)
    x = rng.standard_normal((300, D))
    pi = orot.rotation_seeded(1, 1, 1, D)
    codes, _ = polar.encode(x, pi, bits)
    y = x @ pi.T
    u = y / np.linalg.norm(y, axis=1, keepdims=True)
    err = np.linalg.norm(polar.direction(codes, bits) - u, axis=1)
    bound = np.pi / (1 << bits) + 6 * np.pi / (1 << (bits + 2))
    assert np.all(err <= bound)
    # more bits, less error
    if bits > 2:
        c2, _ = polar.encode(x, pi, bits - 1)
        e2 = np.linalg.norm(polar.direction(c2, bits - 1) - u, axis=1)
        assert err.mean() < e2.mean()


def test_higher_level_angles_concentrate():
    # [P3]: angles of random high-dimensional vectors concentrate; the level-l angle of
    # a rotated Gaussian vector compares two norms of 2^(l-1) coordinates each, so it
    # centres on pi/4 with a spread that shrinks level by level
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4000, D))
    ang, rad = polar.polar_angles(x @ orot.rotation_seeded(1, 3, 0, D).T)
    spreads = [np.std(a) for a in ang[1:]]
    assert all(s1 > s2 for s1, s2 in zip(spreads, spreads[1:]))
    assert all(abs(np.mean(a) - np.pi / 4) < 0.01 for a in ang[1:])
    assert np.allclose(rad, np.linalg.norm(x, axis=1), rtol=1e-12)


def test_page_layout_round_trip():
    assert [polar.page_bytes(D, b) for b in (4, 3, 2)] == [1056, 800, 544]
    # [P3]: the only per-vector constant is the 2-byte radius
    assert polar.page_bytes(D, 3) // 16 - pack.record_bytes(D, 3) == 2
    rng = np.random.default_rng(8)
    nb, hkv, bits = 3, 2, 3
    pool = np.full(nb * hkv * polar.page_bytes(D, bits), 0xA5, np.uint8)
    codes = rng.integers(0, 8, size=(5, D))
    r = np.array([1.0, 0.5, 65504.0, 0.0, 3.140625])
    slots = np.array([0, 17, 33, -1, 47])
    polar.write_pages(pool, slots, 1, hkv, D, bits, codes, r)
    pages = pack.pool_pages(pool, nb, hkv, polar.page_bytes(D, bits))
    c, rr = polar.split_pages(pages, D, bits)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(c[s // 16, 1, s % 16], codes[i]) and rr[s // 16, 1, s % 16] == r[i]
    assert np.all(pages[:, 0] == 0xA5)  # head 0 untouched
    # radius bytes: little-endian fp16 right after the 16 records
    off = 16 * pack.record_bytes(D, bits)
    assert bytes(pages[2, 1, off + 2 * 15: off + 2 * 16]) == np.float16(3.140625).tobytes()


def test_attention_one_token_and_identical_keys():
    rng = np.random.default_rng(9)
    bits, nb, hkv = 4, 4, 1
    pb = polar.page_bytes(D, bits)
    kpool = np.zeros(nb * pb, np.uint8)
    vpool = np.zeros(nb * pb, np.uint8)
    pi = orot.rotation_seeded(1, 2, 0, D)
    k = rng.standard_normal((20, D))
    v = rng.standard_normal((20, D))
    kc, kr = polar.encode(k, pi, bits)
    vc, vr = polar.encode(v, pi, bits)
    bt = np.array([[2, 0]], np.int32)
    slots = np.concatenate([2 * 16 + np.arange(16), np.arange(4)])
    polar.write_pages(kpool, slots, 0, hkv, D, bits, kc, kr)
    polar.write_pages(vpool, slots, 0, hkv, D, bits, vc, vr)
    q = rng.standard_normal((1, 2, D))
    out = polar.decode_attention(q, kpool, vpool, pi, bits, bits, nb, hkv, bt, np.array([1]), 0.1)
    v_hat = polar.decode(vc[:1], vr[:1], pi, bits)[0]
    assert np.allclose(out[0, 0], v_hat, atol=1e-13) and np.allclose(out[0, 1], v_hat, atol=1e-13)
    # identical keys: the mean of the decoded values
    kc2 = np.repeat(kc[:1], 20, axis=0)
    kr2 = np.repeat(kr[:1], 20)
    polar.write_pages(kpool, slots, 0, hkv, D, bits, kc2, kr2)
    out = polar.decode_attention(q, kpool, vpool, pi, bits, bits, nb, hkv, bt, np.array([20]), 0.1)
    assert np.allclose(out[0, 0], polar.decode(vc, vr, pi, bits).mean(axis=0), atol=1e-12)
