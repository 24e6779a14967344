"""Pins for packing and the page layout (CPU only)."""
import os
import struct

import numpy as np
import pytest

import workloads
from oracle import pack

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "p4_pack_example.txt")


def read_golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":" if ":" in line and "=" not in line else "=")
            out[key.strip()] = val.strip()
    return out


def test_page_worked_example():
    """The qiita page's worked example: eight 4-bit codes packed two per byte and
    the scale 0.125 as a little-endian fp32 give the printed bytes, and the two
    bf16 values give theirs."""
    g = read_golden()
    codes = [int(v) for v in g["codes"].split()]
    scale = float(g["scale"])
    packed4 = pack.pack_bits(codes, 4) + struct.pack("<f", scale)
    bf16 = workloads.bf16_bits(np.array([float(v) for v in g["bf16_values"].split()], np.float32))
    assert packed4.hex() == g["packed4"]
    assert bf16.astype("<u2").tobytes().hex() == g["bf16"]
    assert len(packed4) + 2 * bf16.size == int(g["payload_bytes"])
    assert pack.unpack_bits(packed4[:4], 4, 8) == codes


def test_page_example_through_the_pool_layout():
    """The example's record written into a guard-filled pool with the oracle's
    own page arithmetic: the code bytes and the scale land at the record's and
    the norm's places with the printed bytes, a save / clear / restore of
    exactly those two ranges reproduces them, and every other byte of the pool
    keeps the guard fill."""
    g = read_golden()
    codes = [int(v) for v in g["codes"].split()]
    scale = float(g["scale"])
    fill = int(g["fill"], 16)
    d, bits, heads, nblocks = len(codes), 4, 2, 3
    pb = pack.page_bytes(d, bits)
    pool = np.full(nblocks * heads * pb, fill, dtype=np.uint8)
    slot, head = 1 * pack.BLOCK + 7, 1
    pack.write_record(pool, slot, head, heads, d, bits, codes, scale)
    base = pack.page_offset(slot // pack.BLOCK, head, heads, pb)
    tok, rb = slot % pack.BLOCK, pack.record_bytes(d, bits)
    ranges = [(base + tok * rb, rb), (base + pack.BLOCK * rb + 4 * tok, 4)]
    written = b"".join(pool[o:o + n].tobytes() for o, n in ranges)
    assert written.hex() == g["packed4"]
    saved = [pool[o:o + n].copy() for o, n in ranges]
    for o, n in ranges:
        pool[o:o + n] = 0
    for (o, n), data in zip(ranges, saved):
        pool[o:o + n] = data
    assert pack.read_record(pool, slot, head, heads, d, bits) == (codes, scale)
    untouched = np.ones(pool.size, bool)
    for o, n in ranges:
        untouched[o:o + n] = False
    assert np.all(pool[untouched] == fill)


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 8])
def test_round_trip_and_vectorised_agree(bits):
    g = np.random.default_rng(bits)
    codes = g.integers(0, 1 << bits, size=(5, 128))
    for row in codes:
        assert pack.unpack_bits(pack.pack_bits(row, bits), bits, 128) == list(row)
    rec = pack.pack_records(codes, bits)
    assert rec.shape == (5, 128 * bits // 8)
    assert all(rec[i].tobytes() == pack.pack_bits(codes[i], bits) for i in range(5))
    assert np.array_equal(pack.unpack_records(rec, bits, 128), codes)


def test_lsb_first_three_bit_layout():
    # code j occupies bits [3j, 3j+3): codes 1..8 mod 8 -> hand-computed bytes
    codes = [1, 2, 3, 4, 5, 6, 7, 0]
    bitstr = "".join(format(c, "03b")[::-1] for c in codes)  # LSB first per code
    expect = bytes(int(bitstr[i:i + 8][::-1], 2) for i in range(0, 24, 8))
    assert pack.pack_bits(codes, 3) == expect == bytes([0xD1, 0x58, 0x1F])


def test_write_record_touches_only_its_bytes():
    d, bits, heads, nblocks = 128, 4, 2, 3
    pb = pack.page_bytes(d, bits)
    pool = np.full(nblocks * heads * pb, 0xA5, dtype=np.uint8)
    codes = np.arange(d) % 16
    pack.write_record(pool, slot=1 * 16 + 5, head=1, num_kv_heads=heads, d=d, bits=bits, codes=codes, gamma=2.5)
    base = (1 * heads + 1) * pb
    changed = np.nonzero(pool != 0xA5)[0]
    rec = set(range(base + 5 * 64, base + 6 * 64)) | set(range(base + 1024 + 20, base + 1024 + 24))
    assert set(changed.tolist()) <= rec
    c, gm = pack.read_record(pool, 21, 1, heads, d, bits)
    assert c == list(codes) and gm == 2.5


def test_page_sizes_and_ratios_from_the_pages():
    d = 128
    # 4-bit record + fp32 norm = 68 B/vector -> 256/68 = 3.765x (turboquant-vllm
    # "Results": 1,639 MiB -> 435 MiB = 3.76x), 4.25 bits/coord (turbo4, 3.8x)
    rec4 = pack.record_bytes(d, 4) + 4
    assert rec4 == 68
    assert abs(256 / rec4 - 1639 / 435) < 0.01
    assert rec4 * 8 / d == 4.25 and round(16 / 4.25, 1) == 3.8
    # 3-bit keys and values: 3.25 bits -> 4.9x (3bit_nc); k8v4: (8 + 4.25)/2 -> 2.6x
    rec3 = pack.record_bytes(d, 3) + 4
    assert round(16 / (rec3 * 8 / d), 1) == 4.9
    assert round(16 / ((8 + 4.25) / 2), 1) == 2.6
    assert pack.page_bytes(d, 4) == 1088 and pack.page_bytes(d, 3) == 832
    assert pack.page_bytes(d, 2, qjl=True) == 512 + 64 + 256 + 64
    # bf16 boundary layers: K + V = 512 B per token and head (layout table on the qiita page)
    assert 2 * pack.bf16_page_bytes(d) // 16 == 512
    # mixed layout: 62 layers, 4 bf16 at 512 B and 58 packed; with our 136 B/token-head
    ratio = 62 * 512 / (4 * 512 + 58 * 2 * rec4)
    assert 3.15 < ratio < 3.23
    # KV-size formula 2 x 1 x 32 x 8 x 128 x 8192 x 2 B ~ 1.1 GB (Llama 3.1 8B, FP16, 8K)
    assert abs(2 * 1 * 32 * 8 * 128 * 8192 * 2 / 1e9 - 1.07) < 0.01
