"""Pins for the oracle's reference decode attention (CPU only)."""
import math

import numpy as np
from scipy import special

from oracle import attention as oa, codebook as cb, pack, quantize as oq, rotation


def build_packed(x_k, x_v, pi, bits_k, bits_v, block_table, ctx, num_blocks, heads):
    """Quantize [B, T, H, d] K/V with the oracle and write them into pools."""
    d = x_k.shape[-1]
    ck, bk = cb.codebook_fp32(d, bits_k)
    cv, bv = cb.codebook_fp32(d, bits_v)
    kp = np.zeros(num_blocks * heads * pack.page_bytes(d, bits_k), np.uint8)
    vp = np.zeros(num_blocks * heads * pack.page_bytes(d, bits_v), np.uint8)
    for b in range(x_k.shape[0]):
        slots = oa.token_slots(block_table[b], ctx)
        for h in range(heads):
            ik, gk, _ = oq.quantize(x_k[b, :ctx, h], pi, ck, bk)
            iv, gv, _ = oq.quantize(x_v[b, :ctx, h], pi, cv, bv)
            for t in range(ctx):
                pack.write_record(kp, int(slots[t]), h, heads, d, bits_k, ik[t], gk[t])
                pack.write_record(vp, int(slots[t]), h, heads, d, bits_v, iv[t], gv[t])
    return kp, vp, oa.PackedLayer(pi, ck, cv, bits_k, bits_v)


def test_single_token_returns_value():
    d = 128
    g = np.random.default_rng(0)
    k = g.standard_normal((1, 16, 1, d))
    v = g.standard_normal((1, 16, 1, d))
    pi = rotation.hadamard_rotation_seeded(0, 0, d)
    bt = np.array([[2]], np.int32)
    kp, vp, layer = build_packed(k, v, pi, 4, 4, bt, 1, 3, 1)
    q = g.standard_normal((1, 1, d))
    out = oa.decode_packed(q, kp, vp, layer, 3, 1, bt, [1], 1 / math.sqrt(d))
    f = oa.gather_packed(kp, vp, layer, 3, 1, d, bt[0], 1, 0)
    assert np.allclose(out[0, 0], f["v_hat"][0], atol=1e-14)


def test_identical_keys_average_values():
    d, t = 128, 37
    g = np.random.default_rng(1)
    k = np.repeat(g.standard_normal((1, 1, 1, d)), t, axis=1)
    v = g.standard_normal((1, t, 1, d))
    pi = rotation.hadamard_rotation_seeded(0, 1, d)
    bt = np.array([[4, 0, 2]], np.int32)
    kp, vp, layer = build_packed(k, v, pi, 3, 4, bt, t, 5, 1)
    q = g.standard_normal((1, 2, d))  # two query heads share the one KV head
    out = oa.decode_packed(q, kp, vp, layer, 5, 1, bt, [t], 0.3)
    f = oa.gather_packed(kp, vp, layer, 5, 1, d, bt[0], t, 0)
    assert np.allclose(out[0, 0], f["v_hat"].mean(axis=0), atol=1e-13)
    assert np.allclose(out[0, 1], f["v_hat"].mean(axis=0), atol=1e-13)


def test_textbook_softmax_attention():
    g = np.random.default_rng(2)
    q, k, v = g.standard_normal(8), g.standard_normal((5, 8)), g.standard_normal((5, 8))
    ref = special.softmax(0.7 * (k @ q)) @ v
    assert np.allclose(oa.softmax_attention(q, k, v, 0.7), ref, atol=1e-15)
    # two tokens by hand: weights 1/(1+e^{-delta}), e^{-delta}/(1+e^{-delta})
    k2 = np.array([[1.0, 0.0], [0.0, 1.0]])
    v2 = np.array([[2.0, 0.0], [0.0, 4.0]])
    q2 = np.array([3.0, 1.0])
    w0 = 1.0 / (1.0 + math.exp(-2.0))
    assert np.allclose(oa.softmax_attention(q2, k2, v2, 1.0), [2 * w0, 4 * (1 - w0)], atol=1e-15)


def test_identity_rotation_is_plain_attention_over_dequantized():
    d, t = 128, 40
    g = np.random.default_rng(3)
    k = g.standard_normal((1, t, 1, d))
    v = g.standard_normal((1, t, 1, d))
    bt = np.array([[0, 1, 2]], np.int32)
    kp, vp, layer = build_packed(k, v, np.eye(d), 4, 4, bt, t, 3, 1)
    q = g.standard_normal((1, 1, d))
    out = oa.decode_packed(q, kp, vp, layer, 3, 1, bt, [t], 0.1)
    ck, _ = cb.codebook_fp32(d, 4)
    f = oa.gather_packed(kp, vp, layer, 3, 1, d, bt[0], t, 0)
    khat = ck[f["k_idx"]] * f["k_gamma"][:, None]
    vhat = ck[f["v_idx"]] * f["v_gamma"][:, None]
    ref = special.softmax(0.1 * khat @ q[0, 0]) @ vhat
    assert np.allclose(out[0, 0], ref, atol=1e-13)
    # and it approximates unquantized attention (4-bit: cosine > 0.99)
    exact = special.softmax(0.1 * k[0, :, 0] @ q[0, 0]) @ v[0, :, 0]
    assert np.dot(out[0, 0], exact) / np.linalg.norm(out[0, 0]) / np.linalg.norm(exact) > 0.99


def test_bf16_layer_and_empty_context():
    import workloads
    d, heads, nb = 128, 2, 4
    g = np.random.default_rng(4)
    kf = g.standard_normal((nb, heads, 16, d)).astype(np.float32)
    vf = g.standard_normal((nb, heads, 16, d)).astype(np.float32)
    kb, vb = workloads.bf16_bits(kf), workloads.bf16_bits(vf)
    bt = np.array([[3, 1], [0, 2]], np.int32)
    q = g.standard_normal((2, 4, d))
    out = oa.decode_bf16(q, kb, vb, nb, heads, bt, [20, 0], 0.2)
    kk = workloads.bf16_to_f32(kb).astype(np.float64)
    vv = workloads.bf16_to_f32(vb).astype(np.float64)
    keys = np.concatenate([kk[3, 1], kk[1, 1, :4]])
    vals = np.concatenate([vv[3, 1], vv[1, 1, :4]])
    assert np.allclose(out[0, 3], special.softmax(0.2 * keys @ q[0, 3]) @ vals, atol=1e-13)
    assert np.all(out[1] == 0.0)


def test_k8v4_layer_is_plain_attention_over_fp8_keys():
    """k8v4 pools built by hand (FP8 key records, 4-bit value records): the oracle's
    decode equals scipy softmax attention of the raw query against the FP8-decoded
    keys, with the decoded values; the gather returns the written key bytes."""
    from oracle import fp8
    d, heads, ctx, nb = 128, 2, 37, 5
    g = np.random.default_rng(12)
    pi = rotation.hadamard_rotation_seeded(4, 2, d)
    bt = np.array([[3, 0, 4]], np.int32)
    xk = g.standard_normal((1, 48, heads, d)) * 3.0
    xv = g.standard_normal((1, 48, heads, d))
    cv, bv = cb.codebook_fp32(d, 4)
    kp = np.zeros(nb * heads * fp8.page_bytes(d), np.uint8)
    vp = np.zeros(nb * heads * pack.page_bytes(d, 4), np.uint8)
    slots = oa.token_slots(bt[0], ctx)
    kbytes = fp8.encode(xk[0, :ctx])  # [ctx, heads, d]
    for h in range(heads):
        iv, gv, _ = oq.quantize(xv[0, :ctx, h], pi, cv, bv)
        for t in range(ctx):
            s = int(slots[t])
            o = pack.page_offset(s // 16, h, heads, fp8.page_bytes(d)) + (s % 16) * d
            kp[o: o + d] = kbytes[t, h]
            pack.write_record(vp, s, h, heads, d, 4, iv[t], gv[t])
    layer = oa.PackedLayer(pi, cv, cv, 4, 4)
    q = g.standard_normal((1, 4, d))
    out = oa.decode_k8v4(q, kp, vp, layer, nb, heads, bt, np.array([ctx]), 0.1)
    for h in range(heads):
        k, v = oa.gather_k8v4(kp, vp, layer, nb, heads, d, bt[0], ctx, h)
        assert np.array_equal(fp8.encode(k), kbytes[:, h])
        iv, gv, _ = oq.quantize(xv[0, :ctx, h], pi, cv, bv)
        g32 = gv.astype(np.float32).astype(np.float64)  # the page holds gamma in fp32
        assert np.allclose(v, oq.dequantize(iv, g32, pi, cv), rtol=0, atol=1e-12)
        for hq in (2 * h, 2 * h + 1):
            ref = special.softmax(0.1 * (fp8.decode(kbytes[:, h]) @ q[0, hq])) @ v
            assert np.allclose(out[0, hq], ref, rtol=1e-12, atol=1e-12)
