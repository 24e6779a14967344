"""Seeded synthetic inputs shared by the tests, the bench and the oracle.

This module only draws and lays out input data (K/V vectors, queries, block
tables, slot mappings).  It holds none of the method's arithmetic, so both the
CUDA path and the oracle may take their inputs from it.

Recipes (shapes and value distributions of the workloads the pages describe):

* tiny       : 1 seq, 1 KV head, d = 128, 256 tokens; K, V fp32 iid N(0, 1)
               with 4 outlier channels (drawn without replacement from the
               seed) scaled x20; q N(0, 1).
* llama8b    : batch 16, 32 query / 8 KV heads, d = 128, context 8192; bf16
               K/V = N(0, 1) * s[head, channel], s ~ lognormal(0, 1); paged
               16-token blocks under a shuffled block table.
* long70b    : batch 4, 64 query / 8 KV heads, context 131072; bf16 K/V
               N(0, 1) where each element is replaced with probability 0.01 by
               an (unscaled) Student-t(3) draw.
* vlm_burst  : 36 layers x 8 KV heads, 11,000 prefilled tokens of bf16 K/V
               N(0, 1) * lambda_layer, lambda_layer ~ U(0.5, 4); then decode at
               batch 1 with 32 query heads.
* mixed62    : 62 layers (layers 0, 1, 60, 61 bf16, the rest packed 4-bit),
               8 KV heads, 32 query heads, batch 8, context 100,000; bf16 N(0, 1).

bf16 values are produced by round-to-nearest-even of fp32 draws and returned
as uint16 bit patterns.
"""

import numpy as np

BLOCK = 16


def rng(seed):
    return np.random.Generator(np.random.PCG64(int(seed)))


def bf16_bits(x):
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_f32(u16):
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- K/V draws

def tiny_kv(seed=0, n_tokens=256, d=128, n_outliers=4, scale=20.0):
    """Returns (k, v, q, outlier_channels); k, v fp32 [n_tokens, 1, d], q fp32 [1, 1, d]."""
    g = rng(seed)
    ch = g.choice(d, size=n_outliers, replace=False)
    k = g.standard_normal((n_tokens, 1, d)).astype(np.float32)
    v = g.standard_normal((n_tokens, 1, d)).astype(np.float32)
    k[..., ch] *= np.float32(scale)
    v[..., ch] *= np.float32(scale)
    q = g.standard_normal((1, 1, d)).astype(np.float32)
    return k, v, q, np.sort(ch)


def lognormal_channel_kv(seed, n_tokens, n_kv_heads, d=128):
    """bf16 bits [n_tokens, H_kv, d] for K and V with per-(head, channel) lognormal scales."""
    g = rng(seed)
    sk = g.lognormal(0.0, 1.0, size=(n_kv_heads, d)).astype(np.float32)
    sv = g.lognormal(0.0, 1.0, size=(n_kv_heads, d)).astype(np.float32)
    k = g.standard_normal((n_tokens, n_kv_heads, d), dtype=np.float32) * sk
    v = g.standard_normal((n_tokens, n_kv_heads, d), dtype=np.float32) * sv
    return bf16_bits(k), bf16_bits(v)


def heavy_tail_kv(seed, n_tokens, n_kv_heads, d=128, p=0.01, df=3):
    g = rng(seed)
    out = []
    for _ in range(2):
        x = g.standard_normal((n_tokens, n_kv_heads, d), dtype=np.float32)
        mask = g.random((n_tokens, n_kv_heads, d)) < p
        x[mask] = g.standard_t(df, size=int(mask.sum())).astype(np.float32)
        out.append(bf16_bits(x))
    return out[0], out[1]


def layer_scales(seed, n_layers, lo=0.5, hi=4.0):
    return rng(seed).uniform(lo, hi, size=n_layers).astype(np.float32)


def scaled_gaussian_kv(seed, n_tokens, n_kv_heads, d=128, scale=1.0):
    g = rng(seed)
    k = g.standard_normal((n_tokens, n_kv_heads, d), dtype=np.float32) * np.float32(scale)
    v = g.standard_normal((n_tokens, n_kv_heads, d), dtype=np.float32) * np.float32(scale)
    return bf16_bits(k), bf16_bits(v)


def queries(seed, batch, n_q_heads, d=128, dtype="bf16"):
    q = rng(seed).standard_normal((batch, n_q_heads, d), dtype=np.float32)
    return bf16_bits(q) if dtype == "bf16" else q


# ------------------------------------------------------ paging (block tables)

def shuffled_block_table(seed, batch, blocks_per_seq, num_blocks=None, shuffle=True):
    """Disjoint physical blocks per sequence, in a random permutation.

    Returns (block_table int32 [batch, blocks_per_seq], num_blocks)."""
    need = batch * blocks_per_seq
    num_blocks = need if num_blocks is None else num_blocks
    if num_blocks < need:
        raise ValueError("not enough blocks")
    perm = rng(seed).permutation(num_blocks)[:need] if shuffle else np.arange(need)
    return perm.reshape(batch, blocks_per_seq).astype(np.int32), num_blocks


def slot_mapping(block_table, positions):
    """Slots for token positions [batch, n] of each sequence -> int64 [batch, n]."""
    bt = np.asarray(block_table, dtype=np.int64)
    pos = np.asarray(positions, dtype=np.int64)
    rows = np.arange(bt.shape[0])[:, None]
    return bt[rows, pos // BLOCK] * BLOCK + pos % BLOCK


def prefill_slots(block_table, ctx):
    """Slots of tokens 0..ctx-1 of every sequence, flattened sequence-major."""
    bsz = np.asarray(block_table).shape[0]
    pos = np.broadcast_to(np.arange(ctx)[None, :], (bsz, ctx))
    return slot_mapping(block_table, pos).reshape(-1)
