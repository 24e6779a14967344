"""Reference decode attention over a paged cache, in fp64.

What decode computes ([P1] §第1段/§第2段 for the cache contents; the paged
block table follows vLLM's PagedAttention, [P1] §起動コマンド):
for every sequence b and query head h (KV head h // g, g = H_q / H_kv),

    k_hat_t = gamma_t Pi^T c_K[idx_t]          (decoded key of token t)
    v_hat_t = gamma'_t Pi^T c_V[idx'_t]        (decoded value of token t)
    s_t     = sm_scale * <q, k_hat_t>          (QJL keys: the unbiased estimate)
    out     = sum_t softmax(s)_t v_hat_t,      t < context_len[b]

with token t of sequence b stored at slot block_table[b][t // 16] * 16 + t % 16.
bf16 layers ([P1] §起動コマンド: first/last two layers kept at full precision;
[P4] layout table: 512 B/token/head) use the raw bf16 K and V.  k8v4 layers
([P1] §プリセット: FP8 keys, 4-bit values) use the FP8 E4M3 keys as stored
(no rotation) with the raw query, and the decoded 4-bit values.

This is exact softmax attention (max-subtracted, one pass over all tokens), no
online/split evaluation.  Pinned by (tests/test_oracle_attention.py): one token
gives o = v_hat; identical keys give the mean of v_hat; Pi = I and 8-bit
codebook-free raw bf16 reduce to scipy.special.softmax attention; a
hand-computed two-token case; the k8v4 gather returns exactly the encoded
keys and the decoded values of the records it was handed.
"""

import numpy as np

from . import fp8, pack, qjl as qjl_mod
from .quantize import bf16_bits_to_f64


def softmax_attention(q, k, v, sm_scale):
    """q [d], k [T, d], v [T, d] -> [d]; exact softmax in fp64."""
    q = np.asarray(q, dtype=np.float64)
    s = sm_scale * (np.asarray(k, dtype=np.float64) @ q)
    return softmax_weights(s) @ np.asarray(v, dtype=np.float64)


def softmax_weights(s):
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - np.max(s))
    return e / np.sum(e)


def token_slots(block_table_row, ctx):
    t = np.arange(ctx)
    blocks = np.asarray(block_table_row, dtype=np.int64)[t // pack.BLOCK]
    return blocks * pack.BLOCK + t % pack.BLOCK


class PackedLayer:
    """Everything the oracle needs to decode one packed layer."""

    def __init__(self, pi, cb_k, cb_v, bits_k, bits_v, qjl_s=None):
        self.pi = np.asarray(pi, dtype=np.float64)
        self.cb_k = np.asarray(cb_k, dtype=np.float64)
        self.cb_v = np.asarray(cb_v, dtype=np.float64)
        self.bits_k = bits_k
        self.bits_v = bits_v
        self.qjl_s = None if qjl_s is None else np.asarray(qjl_s, dtype=np.float64)

    @property
    def qjl(self):
        return self.qjl_s is not None


def gather_packed(k_pool, v_pool, layer, num_blocks, num_kv_heads, d, block_table_row, ctx, head):
    """Decode the context of one (sequence, kv head) from packed pools.

    Returns dict with rotated-domain fields and decoded k_hat, v_hat [ctx, d].
    """
    m = d
    pbk = pack.page_bytes(d, layer.bits_k, layer.qjl, m)
    pbv = pack.page_bytes(d, layer.bits_v)
    kp = pack.pool_pages(k_pool, num_blocks, num_kv_heads, pbk)
    vp = pack.pool_pages(v_pool, num_blocks, num_kv_heads, pbv)
    slots = token_slots(block_table_row, ctx)
    blocks = slots // pack.BLOCK
    toks = slots % pack.BLOCK
    kf = pack.split_pages(kp[blocks, head], d, layer.bits_k, layer.qjl, m)
    vf = pack.split_pages(vp[blocks, head], d, layer.bits_v)
    sel = np.arange(ctx)
    k_idx = kf[0][sel, toks]
    k_gamma = kf[1][sel, toks]
    v_idx = vf[0][sel, toks]
    v_gamma = vf[1][sel, toks]
    out = {
        "k_idx": k_idx, "k_gamma": k_gamma, "v_idx": v_idx, "v_gamma": v_gamma,
        "k_hat": (layer.cb_k[k_idx] * k_gamma[:, None]) @ layer.pi,
        "v_hat": (layer.cb_v[v_idx] * v_gamma[:, None]) @ layer.pi,
    }
    if layer.qjl:
        out["k_signs"] = kf[2][sel, toks]
        out["k_rho"] = kf[3][sel, toks]
    return out


def decode_packed(q, k_pool, v_pool, layer, num_blocks, num_kv_heads, block_table, context_lens, sm_scale):
    """q [B, H_q, d] f64 -> out [B, H_q, d] f64 over a packed layer."""
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    g = hq // num_kv_heads
    out = np.zeros_like(q)
    for b in range(bsz):
        ctx = int(context_lens[b])
        if ctx == 0:
            continue
        for kvh in range(num_kv_heads):
            f = gather_packed(k_pool, v_pool, layer, num_blocks, num_kv_heads, d, block_table[b], ctx, kvh)
            for h in range(kvh * g, (kvh + 1) * g):
                if layer.qjl:
                    s = sm_scale * qjl_mod.estimate(q[b, h], layer.pi, layer.cb_k, f["k_idx"], f["k_gamma"],
                                                    f["k_signs"], f["k_rho"], layer.qjl_s)
                else:
                    s = sm_scale * (f["k_hat"] @ q[b, h])
                out[b, h] = softmax_weights(s) @ f["v_hat"]
    return out


def gather_bf16(k_pool_u16, v_pool_u16, num_blocks, num_kv_heads, d, block_table_row, ctx, head):
    """Raw bf16 K/V of one (sequence, kv head) as fp64 [ctx, d]."""
    kp = np.asarray(k_pool_u16, dtype=np.uint16).reshape(num_blocks, num_kv_heads, pack.BLOCK, d)
    vp = np.asarray(v_pool_u16, dtype=np.uint16).reshape(num_blocks, num_kv_heads, pack.BLOCK, d)
    slots = token_slots(block_table_row, ctx)
    blocks = slots // pack.BLOCK
    toks = slots % pack.BLOCK
    return bf16_bits_to_f64(kp[blocks, head, toks]), bf16_bits_to_f64(vp[blocks, head, toks])


def decode_bf16(q, k_pool_u16, v_pool_u16, num_blocks, num_kv_heads, block_table, context_lens, sm_scale):
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    g = hq // num_kv_heads
    out = np.zeros_like(q)
    for b in range(bsz):
        ctx = int(context_lens[b])
        if ctx == 0:
            continue
        for kvh in range(num_kv_heads):
            k, v = gather_bf16(k_pool_u16, v_pool_u16, num_blocks, num_kv_heads, d, block_table[b], ctx, kvh)
            for h in range(kvh * g, (kvh + 1) * g):
                out[b, h] = softmax_attention(q[b, h], k, v, sm_scale)
    return out


def gather_k8v4(k_pool, v_pool, layer, num_blocks, num_kv_heads, d, block_table_row, ctx, head):
    """One (sequence, kv head) of a k8v4 layer: FP8 E4M3 keys as stored (no rotation,
    no scale) and the 4-bit (bits_v) TurboQuant values decoded to x_hat; [ctx, d] each."""
    kp = pack.pool_pages(k_pool, num_blocks, num_kv_heads, fp8.page_bytes(d))
    vp = pack.pool_pages(v_pool, num_blocks, num_kv_heads, pack.page_bytes(d, layer.bits_v))
    slots = token_slots(block_table_row, ctx)
    blocks = slots // pack.BLOCK
    toks = slots % pack.BLOCK
    krec = kp[blocks, head].reshape(ctx, pack.BLOCK, d)[np.arange(ctx), toks]
    vf = pack.split_pages(vp[blocks, head], d, layer.bits_v)
    sel = np.arange(ctx)
    v_idx = vf[0][sel, toks]
    v_gamma = vf[1][sel, toks]
    return fp8.decode(krec), (layer.cb_v[v_idx] * v_gamma[:, None]) @ layer.pi


def decode_k8v4(q, k_pool, v_pool, layer, num_blocks, num_kv_heads, block_table, context_lens, sm_scale):
    """q [B, H_q, d] f64 -> out [B, H_q, d] f64 over a k8v4 layer: exact softmax
    attention of the raw query against the FP8 keys, values from their codes."""
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    g = hq // num_kv_heads
    out = np.zeros_like(q)
    for b in range(bsz):
        ctx = int(context_lens[b])
        if ctx == 0:
            continue
        for kvh in range(num_kv_heads):
            k, v = gather_k8v4(k_pool, v_pool, layer, num_blocks, num_kv_heads, d, block_table[b], ctx, kvh)
            for h in range(kvh * g, (kvh + 1) * g):
                out[b, h] = softmax_attention(q[b, h], k, v, sm_scale)
    return out
