"""Pins of the oracle's cache images (offload / restore)."""
import numpy as np

from oracle import offload


def test_fnv1a64_known_answers():
    # published test vectors of FNV-1a 64
    assert offload.fnv1a64(b"") == 0xCBF29CE484222325
    assert offload.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert offload.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_header_round_trip():
    h = offload.header((0, 4, 3, 1, 2, 0), 128, 8, 16, 37, 0x0123456789ABCDEF)
    assert len(h) == offload.HEADER
    p = offload.parse_header(h)
    assert p["fmt"] == (0, 4, 3, 1, 2, 0) and p["n_blocks"] == 37 and p["codebook_hash"] == 0x0123456789ABCDEF
    assert (p["head_dim"], p["num_kv_heads"], p["block_size"], p["version"]) == (128, 8, 16, 1)


def test_image_is_the_listed_pages_in_order():
    g = np.random.default_rng(1)
    nb, H, pk, pv = 9, 2, 48, 32
    kp = g.integers(0, 256, nb * H * pk, dtype=np.uint8)
    vp = g.integers(0, 256, nb * H * pv, dtype=np.uint8)
    blocks = [7, 2, 3, 8]
    head = offload.header((0, 4, 4, 0, 1, 0), 128, H, 16, len(blocks), 5)
    img = offload.build_image(kp, vp, nb, H, pk, pv, blocks, head)
    assert img.size == offload.HEADER + len(blocks) * H * (pk + pv)
    ki, vi = offload.image_pages(img, H, pk, pv)
    for i, b in enumerate(blocks):
        assert np.array_equal(ki[i], kp[b * H * pk:(b + 1) * H * pk])
        assert np.array_equal(vi[i], vp[b * H * pv:(b + 1) * H * pv])
    # pages of unlisted blocks never enter the image: changing them changes nothing
    kp2 = kp.copy()
    kp2[0: H * pk] ^= 0xFF
    assert np.array_equal(offload.build_image(kp2, vp, nb, H, pk, pv, blocks, head), img)
