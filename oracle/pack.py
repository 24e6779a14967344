"""Bit packing of codes and the paged cache layout.

[P4] "4bitという名前だけでは、コピーするサイズは決まらない": the storage dtype
(uint8 containers) is not the value bit width; two 4-bit codes share a byte and
the packed region also carries the scale.  [P4] "小さな保存・復元コードで…":
the worked example packs codes[i] | codes[i+1] << 4 and appends the scale as a
little-endian fp32.

Readings (fixed in include/tq.h):
* Record of one vector: LSB-first bitstream, code j in bits [b*j, b*j + b),
  bit k of the record = bit (k mod 8) of byte (k div 8).  For b = 4 this is
  exactly the page's codes[i] | codes[i+1] << 4.
* Page of one (block, kv_head), block_size 16 tokens:
    [16 x code record (d*b/8 B)] [16 x fp32 gamma]
    (+ keys with QJL: [16 x sign record (m/8 B)] [16 x fp32 rho])
* bf16 page: [16 tokens][d] bf16, row-major.
* Pool: [num_blocks][num_kv_heads][page_bytes]; slot s = block * 16 + offset.

Pinned by (tests/test_oracle_pack.py): the page's worked example bytes
(tests/golden/p4_pack_example.txt), unpack(pack(x)) = x for b in {1..8},
0xA5 guard bytes untouched around written regions.
"""

import numpy as np

BLOCK = 16


def pack_bits(codes, bits):
    """LSB-first bitstream of integer codes, returned as uint8 bytes."""
    codes = [int(v) for v in codes]
    total = len(codes) * bits
    out = bytearray((total + 7) // 8)
    pos = 0
    for v in codes:
        if v < 0 or v >= (1 << bits):
            raise ValueError("code out of range")
        for k in range(bits):
            if (v >> k) & 1:
                out[(pos + k) // 8] |= 1 << ((pos + k) % 8)
        pos += bits
    return bytes(out)


def unpack_bits(data, bits, count):
    data = bytes(data)
    out = []
    pos = 0
    for _ in range(count):
        v = 0
        for k in range(bits):
            if (data[(pos + k) // 8] >> ((pos + k) % 8)) & 1:
                v |= 1 << k
        out.append(v)
        pos += bits
    return out


def record_bytes(d, bits):
    return d * bits // 8


def page_bytes(d, bits, qjl=False, m=None):
    n = BLOCK * record_bytes(d, bits) + BLOCK * 4
    if qjl:
        m = d if m is None else m
        n += BLOCK * (m // 8) + BLOCK * 4
    return n


def bf16_page_bytes(d):
    return BLOCK * d * 2


def page_offset(block, head, num_kv_heads, pbytes):
    return (block * num_kv_heads + head) * pbytes


def write_record(pool, slot, head, num_kv_heads, d, bits, codes, gamma,
                 qjl_signs=None, rho=None, m=None):
    """Write one vector's record into a uint8 pool (numpy array) in place."""
    qjl = qjl_signs is not None
    pb = page_bytes(d, bits, qjl, m)
    base = page_offset(slot // BLOCK, head, num_kv_heads, pb)
    tok = slot % BLOCK
    rb = record_bytes(d, bits)
    pool[base + tok * rb: base + (tok + 1) * rb] = np.frombuffer(pack_bits(codes, bits), dtype=np.uint8)
    goff = base + BLOCK * rb + 4 * tok
    pool[goff:goff + 4] = np.frombuffer(np.float32(gamma).tobytes(), dtype=np.uint8)
    if qjl:
        m = d if m is None else m
        sb = m // 8
        soff = base + BLOCK * rb + BLOCK * 4 + tok * sb
        pool[soff:soff + sb] = np.frombuffer(pack_bits(qjl_signs, 1), dtype=np.uint8)
        roff = base + BLOCK * rb + BLOCK * 4 + BLOCK * sb + 4 * tok
        pool[roff:roff + 4] = np.frombuffer(np.float32(rho).tobytes(), dtype=np.uint8)


def read_record(pool, slot, head, num_kv_heads, d, bits, qjl=False, m=None):
    """Returns (codes list, gamma f64[, signs list, rho f64])."""
    pool = np.asarray(pool, dtype=np.uint8)
    pb = page_bytes(d, bits, qjl, m)
    base = page_offset(slot // BLOCK, head, num_kv_heads, pb)
    tok = slot % BLOCK
    rb = record_bytes(d, bits)
    codes = unpack_bits(pool[base + tok * rb: base + (tok + 1) * rb].tobytes(), bits, d)
    goff = base + BLOCK * rb + 4 * tok
    gamma = float(np.frombuffer(pool[goff:goff + 4].tobytes(), dtype="<f4")[0])
    if not qjl:
        return codes, gamma
    m = d if m is None else m
    sb = m // 8
    soff = base + BLOCK * rb + BLOCK * 4 + tok * sb
    signs = unpack_bits(pool[soff:soff + sb].tobytes(), 1, m)
    roff = base + BLOCK * rb + BLOCK * 4 + BLOCK * sb + 4 * tok
    rho = float(np.frombuffer(pool[roff:roff + 4].tobytes(), dtype="<f4")[0])
    return codes, gamma, signs, rho


def read_page_codes(pool, block, head, num_kv_heads, d, bits, qjl=False, m=None):
    """Vectorised reader for a whole page: (codes [16, d], gamma [16][, signs [16, m], rho [16]])."""
    out = [read_record(pool, block * BLOCK + t, head, num_kv_heads, d, bits, qjl, m) for t in range(BLOCK)]
    codes = np.array([o[0] for o in out], dtype=np.int64)
    gamma = np.array([o[1] for o in out], dtype=np.float64)
    if not qjl:
        return codes, gamma
    signs = np.array([o[2] for o in out], dtype=np.int64)
    rho = np.array([o[3] for o in out], dtype=np.float64)
    return codes, gamma, signs, rho


def unpack_records(records, bits, count):
    """Vectorised unpack_bits over rows of a uint8 array [n, R] -> int64 [n, count].

    np.unpackbits(bitorder="little") lists bit (k mod 8) of byte (k div 8) at
    position k, which is the bitstream order defined above.
    """
    records = np.ascontiguousarray(records, dtype=np.uint8)
    bitsarr = np.unpackbits(records, axis=-1, bitorder="little")[..., : count * bits]
    bitsarr = bitsarr.reshape(records.shape[:-1] + (count, bits)).astype(np.int64)
    weights = (1 << np.arange(bits, dtype=np.int64))
    return (bitsarr * weights).sum(axis=-1)


def pack_records(codes, bits):
    """Vectorised pack_bits over rows of an int array [n, count] -> uint8 [n, R]."""
    codes = np.asarray(codes, dtype=np.int64)
    if codes.size and (codes.min() < 0 or codes.max() >= (1 << bits)):
        raise ValueError("code out of range")
    shifts = np.arange(bits, dtype=np.int64)
    bitsarr = ((codes[..., None] >> shifts) & 1).astype(np.uint8)
    flat = bitsarr.reshape(codes.shape[:-1] + (codes.shape[-1] * bits,))
    return np.packbits(flat, axis=-1, bitorder="little")


def pool_pages(pool, num_blocks, num_kv_heads, pbytes):
    """View a flat uint8 pool as [num_blocks, num_kv_heads, page_bytes]."""
    return np.asarray(pool, dtype=np.uint8).reshape(num_blocks, num_kv_heads, pbytes)


def split_pages(pages, d, bits, qjl=False, m=None):
    """Split pages [..., page_bytes] into their fields.

    Returns (codes [..., 16, d], gamma f64 [..., 16][, signs [..., 16, m], rho [..., 16]]).
    """
    pages = np.asarray(pages, dtype=np.uint8)
    rb = record_bytes(d, bits)
    lead = pages.shape[:-1]
    codes = unpack_records(pages[..., : BLOCK * rb].reshape(lead + (BLOCK, rb)), bits, d)
    g = pages[..., BLOCK * rb: BLOCK * rb + 4 * BLOCK].copy()
    gamma = g.view("<f4").reshape(lead + (BLOCK,)).astype(np.float64)
    if not qjl:
        return codes, gamma
    m = d if m is None else m
    sb = m // 8
    o = BLOCK * rb + 4 * BLOCK
    signs = unpack_records(pages[..., o: o + BLOCK * sb].reshape(lead + (BLOCK, sb)), 1, m)
    r = pages[..., o + BLOCK * sb: o + BLOCK * sb + 4 * BLOCK].copy()
    rho = r.view("<f4").reshape(lead + (BLOCK,)).astype(np.float64)
    return codes, gamma, signs, rho
