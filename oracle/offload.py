"""Host images of cache blocks for offload and restore (test infrastructure: the oracle).

[P4] (LMCache's mixed BF16 / 4-bit KV cache): the offload path copies the
stored bytes of each group uninterpreted -- the packed codes, their scales and
the BF16 layers alike -- and restoring them must give back exactly what was
stored, T(Q(X)) = Q(X); the reader must know the format id and version of what
it reads.  The pages leave the container open; the reading (fixed in
include/tq.h) is:

* a 64-byte little-endian header:
    bytes  0.. 7  magic b"TQKVIMG1"
           8..11  format version (uint32)
          12..35  kv_format, bits_k, bits_v, qjl_k, rot_kind, norm_mode (int32 each)
          36..39  head_dim, 40..43 num_kv_heads, 44..47 block_size (int32)
          48..55  number of blocks n (int64)
          56..63  FNV-1a 64 of the 4 codebook tables as stored in the descriptor
                  (centroids_k[16], boundaries_k[15], centroids_v[16],
                  boundaries_v[15], fp32 little-endian, in that order)
* then the K pages of every KV head of each listed block, in the order listed,
  then the V pages of the same blocks in the same order, byte for byte as in
  the pools (so a run of consecutive block ids is one contiguous range of each
  pool and of the image).

Pinned by tests/test_oracle_offload.py: FNV-1a 64 known answers of the
published function, the header fields read back, and image -> pages -> image
is the identity with the pages of unlisted blocks never read.
"""

import struct

import numpy as np

MAGIC = b"TQKVIMG1"
HEADER = 64
FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3


def fnv1a64(data):
    """FNV-1a, 64-bit (Fowler, Noll, Vo): h = offset; h = (h ^ byte) * prime mod 2^64."""
    h = FNV_OFFSET
    for b in bytes(data):
        h ^= b
        h = (h * FNV_PRIME) & 0xFFFFFFFFFFFFFFFF
    return h


def codebook_hash(centroids_k, boundaries_k, centroids_v, boundaries_v):
    raw = b"".join(np.asarray(t, dtype="<f4").tobytes() for t in (centroids_k, boundaries_k, centroids_v,
                                                                  boundaries_v))
    return fnv1a64(raw)


def header(fmt, head_dim, num_kv_heads, block_size, n_blocks, cb_hash, version=1):
    """fmt: (kv_format, bits_k, bits_v, qjl_k, rot_kind, norm_mode)."""
    return (MAGIC + struct.pack("<I", version) + struct.pack("<6i", *fmt)
            + struct.pack("<3i", head_dim, num_kv_heads, block_size) + struct.pack("<q", n_blocks)
            + struct.pack("<Q", cb_hash))


def parse_header(image):
    b = bytes(image[:HEADER])
    if b[:8] != MAGIC:
        raise ValueError("not a cache image")
    version, = struct.unpack_from("<I", b, 8)
    fmt = struct.unpack_from("<6i", b, 12)
    head_dim, heads, block = struct.unpack_from("<3i", b, 36)
    n, = struct.unpack_from("<q", b, 48)
    h, = struct.unpack_from("<Q", b, 56)
    return {"version": version, "fmt": fmt, "head_dim": head_dim, "num_kv_heads": heads, "block_size": block,
            "n_blocks": n, "codebook_hash": h}


def build_image(k_pool, v_pool, num_blocks, num_kv_heads, page_k, page_v, blocks, head):
    """Image of `blocks` from flat uint8 pools; `head` = the 64 header bytes."""
    kp = np.asarray(k_pool, np.uint8).reshape(num_blocks, num_kv_heads * page_k)
    vp = np.asarray(v_pool, np.uint8).reshape(num_blocks, num_kv_heads * page_v)
    idx = np.asarray(blocks, dtype=np.int64)
    return np.concatenate([np.frombuffer(head, np.uint8), kp[idx].reshape(-1), vp[idx].reshape(-1)])


def image_pages(image, num_kv_heads, page_k, page_v):
    """(k_pages [n, H * page_k], v_pages [n, H * page_v]) of an image."""
    n = parse_header(image)["n_blocks"]
    body = np.asarray(image, np.uint8)[HEADER:]
    nk = n * num_kv_heads * page_k
    return body[:nk].reshape(n, num_kv_heads * page_k), body[nk: nk + n * num_kv_heads * page_v].reshape(
        n, num_kv_heads * page_v)
