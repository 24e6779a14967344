"""GPU parity of the PolarQuant-variant layers (append, dequantize, decode)
against the oracle (oracle/polar.py).

Append: the GPU's angle codes equal the oracle's fp64 codes except where the
oracle's pair lies within tau = 1e-5 (on the unit sphere) of the grid edge
between the two codes, radii within one fp16 step.  Dequantize and decode run
on pages the oracle encoded and packed itself (uploaded byte for byte), so
they are compared with nothing taken from the GPU's own encoder; the end-to-end
tests encode on the GPU and compare with the oracle's encoding of the same
inputs."""
import math

import numpy as np
import pytest

import workloads
from oracle import pack as opack, polar as opolar, quantize as oq, rotation as orot
from tests._gpu_util import D, max_rel_err

pytestmark = pytest.mark.gpu

TAU = 1e-5
TOL_F32 = 2e-3
TOL_BF16 = 5e-3


def pair_values(y):
    """(a, b) of every record slot's pair [n, d - 1] on the unit sphere, from block
    norms (level l pairs two blocks of 2^(l-1) coordinates)."""
    y = y / np.linalg.norm(y, axis=1, keepdims=True)
    A, B = [y[:, 0::2]], [y[:, 1::2]]
    for level in range(2, 8):
        w = 1 << (level - 1)
        nrm = np.sqrt(np.sum(y.reshape(y.shape[0], -1, w) ** 2, axis=-1))
        A.append(nrm[:, 0::2])
        B.append(nrm[:, 1::2])
    return np.concatenate(A, axis=1), np.concatenate(B, axis=1)


def slot_level(s):
    return np.where(s < 64, 1, np.where(s < 96, 2, np.where(s < 112, 3, np.where(
        s < 120, 4, np.where(s < 124, 5, np.where(s < 126, 6, 7))))))


def band_ok(x, pi, bits, codes_gpu, codes_or):
    """Every mismatching angle code is one cell off and its pair sits within TAU of the edge."""
    assert np.all(codes_gpu[:, D - 1] == 0)
    mism = codes_gpu[:, :D - 1] != codes_or[:, :D - 1]
    if not mism.any():
        return 0.0
    y = np.asarray(x, np.float64) @ pi.T
    A, B = pair_values(y)
    v, s = np.nonzero(mism)
    kg, ko = codes_gpu[v, s], codes_or[v, s]
    lev = slot_level(s)
    n = 1 << bits
    hi = np.maximum(kg, ko)
    lo = np.minimum(kg, ko)
    wrap = (lev == 1) & (lo == 0) & (hi == n - 1)
    adjacent = (hi - lo == 1) | wrap
    assert np.all(adjacent), "non-adjacent code mismatch"
    theta_e = np.where(lev == 1, np.where(wrap, 0.0, hi * (2 * np.pi / n)) - np.pi, hi * (np.pi / 2 / n))
    dist = np.abs(B[v, s] * np.cos(theta_e) - A[v, s] * np.sin(theta_e))
    assert np.all(dist <= TAU), "code mismatch outside the edge band (max %.3e)" % dist.max()
    return float(mism.mean())


def radius_ok(r_gpu, r_or):
    step = np.spacing(np.abs(r_or).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(r_gpu - r_or) <= step)


def dev_bf16(cuda, bits):
    return cuda.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(cuda.bfloat16)


def polar_fields(layer, which):
    host = (layer.k_cache if which == 0 else layer.v_cache).cpu().numpy()
    bits = layer.bits_k if which == 0 else layer.bits_v
    pages = opack.pool_pages(host, layer.num_blocks, layer.num_kv_heads, opolar.page_bytes(D, bits))
    return opolar.split_pages(pages, D, bits), pages


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_polar_append_matches_oracle(cuda, tqlib, bits, dtype):
    """2001 tokens x 4 KV heads of K and V (8004 vectors each: many warps and a ragged
    tail), every 37th slot skipped; unaddressed records keep their guard bytes."""
    tq = tqlib
    H, n = 4, 2001
    nb = n // 16 + 4
    layer = tq.Layer(nb, H, kv_format="polar", bits_k=bits, bits_v=bits, seed=5, layer=2, fill=0xA5)
    kb, vb = workloads.lognormal_channel_kv(3 + bits, n, H, D)
    slots = np.random.default_rng(bits).permutation(nb * 16)[:n].astype(np.int64)
    slots[::37] = -1
    if dtype == "bf16":
        kx, vx = oq.bf16_bits_to_f64(kb), oq.bf16_bits_to_f64(vb)
        layer.append(dev_bf16(cuda, kb), dev_bf16(cuda, vb), cuda.from_numpy(slots).cuda())
    else:
        kx, vx = workloads.bf16_to_f32(kb) * 1.0001, workloads.bf16_to_f32(vb) * 0.9999  # off the bf16 grid
        kx, vx = kx.astype(np.float32), vx.astype(np.float32)
        layer.append(cuda.from_numpy(kx).cuda(), cuda.from_numpy(vx).cuda(), cuda.from_numpy(slots).cuda())
        kx, vx = kx.astype(np.float64), vx.astype(np.float64)
    assert tq.get_device_status() == 0
    pi = orot.hadamard_rotation_seeded(5, 2, D)
    keep = slots >= 0
    written = np.zeros(nb * 16, bool)
    written[slots[keep]] = True
    rates = []
    for which, x in ((0, kx), (1, vx)):
        (codes, r), pages = polar_fields(layer, which)
        for h in range(H):
            co, ro = opolar.encode(x[keep, h], pi, bits)
            cg = codes[slots[keep] // 16, h, slots[keep] % 16]
            rg = r[slots[keep] // 16, h, slots[keep] % 16]
            rates.append(band_ok(x[keep, h], pi, bits, cg, co))
            radius_ok(rg, ro)
        rb = opack.record_bytes(D, bits)
        recs = pages[:, :, :16 * rb].reshape(nb, H, 16, rb).transpose(0, 2, 1, 3)  # [block, offset, head, byte]
        assert np.all(recs[~written.reshape(nb, 16)] == 0xA5)
    print("edge-band mismatch rate %.2e" % np.mean(rates))
    assert np.mean(rates) < 1e-3


def test_polar_append_zero_vector_and_bad_slot(cuda, tqlib):
    tq = tqlib
    layer = tq.Layer(4, 1, kv_format="polar", bits_k=3, bits_v=3)
    x = np.zeros((2, 1, D), np.float32)
    x[1, 0, 3] = 2.0
    slots = cuda.tensor([5, 4 * 16 + 3], dtype=cuda.int64).cuda()  # the second slot is out of range
    layer.append(cuda.from_numpy(x).cuda(), None, slots)
    assert tq.get_device_status() & tq.TQ_DEV_BAD_SLOT
    assert tq.get_device_status() == 0
    (codes, r), _ = polar_fields(layer, 0)
    co, ro = opolar.encode(np.zeros((1, D)), np.eye(D), 3)  # zero pairs: the same codes under any Pi
    assert np.array_equal(codes[0, 0, 5], co[0]) and r[0, 0, 5] == 0.0


def oracle_pools(seed, nb, H, bits_k, bits_v, pi, kx, vx, slots):
    """Host pools of a polar layer written by the oracle (encode + pack)."""
    kpool = np.zeros(nb * H * opolar.page_bytes(D, bits_k), np.uint8)
    vpool = np.zeros(nb * H * opolar.page_bytes(D, bits_v), np.uint8)
    for h in range(H):
        kc, kr = opolar.encode(kx[:, h], pi, bits_k)
        vc, vr = opolar.encode(vx[:, h], pi, bits_v)
        opolar.write_pages(kpool, slots, h, H, D, bits_k, kc, kr)
        opolar.write_pages(vpool, slots, h, H, D, bits_v, vc, vr)
    return kpool, vpool


def upload(cuda, layer, kpool, vpool):
    layer.k_cache.copy_(cuda.from_numpy(kpool).cuda())
    layer.v_cache.copy_(cuda.from_numpy(vpool).cuda())


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_polar_dequantize_matches_oracle(cuda, tqlib, bits):
    tq = tqlib
    H, n, nb = 3, 700, 50
    layer = tq.Layer(nb, H, kv_format="polar", bits_k=bits, bits_v=5 - bits if bits < 4 else 2, seed=9, layer=1)
    pi = orot.hadamard_rotation_seeded(9, 1, D)
    kb, vb = workloads.scaled_gaussian_kv(bits, n, H, D, scale=3.0)
    kx, vx = oq.bf16_bits_to_f64(kb), oq.bf16_bits_to_f64(vb)
    slots = np.random.default_rng(4).permutation(nb * 16)[:n].astype(np.int64)
    kpool, vpool = oracle_pools(0, nb, H, layer.bits_k, layer.bits_v, pi, kx, vx, slots)
    upload(cuda, layer, kpool, vpool)
    q_slots = slots.copy()
    q_slots[::50] = -1  # negative slots give zero rows
    sd = cuda.from_numpy(q_slots).cuda()
    for which, bw, pool in ((0, layer.bits_k, kpool), (1, layer.bits_v, vpool)):
        pages = opack.pool_pages(pool, nb, H, opolar.page_bytes(D, bw))
        codes, r = opolar.split_pages(pages, D, bw)
        for out_dt, tol in ((cuda.float32, 2e-5), (cuda.bfloat16, 8e-3)):
            out = layer.dequantize(which, sd, out_dtype=out_dt).float().cpu().numpy()
            for h in range(H):
                live = q_slots >= 0
                s = q_slots[live]
                ref = opolar.decode(codes[s // 16, h, s % 16], r[s // 16, h, s % 16], pi, bw)
                assert max_rel_err(out[live, h], ref) <= tol
                assert np.all(out[~live, h] == 0.0)
    assert tq.get_device_status() == 0


def decode_case(cuda, tq, *, B, Hq, Hkv, ctx, bits_k, bits_v, seed=0, num_splits=0, q_f32=False, out_f32=True):
    ctx = np.asarray(ctx, np.int32)
    mb = int(max(1, math.ceil(ctx.max() / 16)))
    bt, nb = workloads.shuffled_block_table(seed + 1, B, mb, num_blocks=B * mb + 3)
    layer = tq.Layer(nb, Hkv, kv_format="polar", bits_k=bits_k, bits_v=bits_v, seed=seed + 7, layer=seed % 5)
    pi = orot.hadamard_rotation_seeded(seed + 7, seed % 5, D)
    kb, vb = workloads.lognormal_channel_kv(seed, B * mb * 16, Hkv, D)
    slots = workloads.prefill_slots(bt, mb * 16)
    kpool, vpool = oracle_pools(seed, nb, Hkv, bits_k, bits_v, pi, oq.bf16_bits_to_f64(kb),
                                oq.bf16_bits_to_f64(vb), slots)
    upload(cuda, layer, kpool, vpool)
    qf = workloads.queries(seed + 3, B, Hq, D, dtype="f32" if q_f32 else "bf16")
    qd = cuda.from_numpy(qf).cuda() if q_f32 else dev_bf16(cuda, qf)
    sm = 1.0 / math.sqrt(D)
    out = layer.decode(qd, cuda.from_numpy(bt).cuda(), cuda.from_numpy(ctx).cuda(), sm_scale=sm,
                       out_dtype=cuda.float32 if out_f32 else cuda.bfloat16, num_splits=num_splits)
    cuda.cuda.synchronize()
    assert tq.get_device_status() == 0
    qx = qf.astype(np.float64) if q_f32 else oq.bf16_bits_to_f64(qf)
    ref = opolar.decode_attention(qx, kpool, vpool, pi, bits_k, bits_v, nb, Hkv, bt, ctx, sm)
    return out.float().cpu().numpy(), ref


@pytest.mark.parametrize("bits_k,bits_v,Hq,Hkv,ctx,splits", [
    (4, 4, 8, 2, [1, 17, 130, 300], 0),       # g = 4, ragged contexts
    (3, 4, 8, 2, [300, 0, 45, 129], 3),       # an empty sequence, odd block counts
    (2, 3, 4, 4, [64, 33], 1),                # g = 1, one split
    (4, 2, 16, 2, [250, 96], 5),              # g = 8
    (4, 4, 12, 1, [200, 31], 2),              # g = 12: head groups of 8 and 4
])
def test_polar_decode_matches_oracle(cuda, tqlib, bits_k, bits_v, Hq, Hkv, ctx, splits):
    out, ref = decode_case(cuda, tqlib, B=len(ctx), Hq=Hq, Hkv=Hkv, ctx=ctx, bits_k=bits_k, bits_v=bits_v,
                           seed=bits_k + 3 * bits_v, num_splits=splits, q_f32=True)
    live = np.asarray(ctx) > 0
    err = max_rel_err(out[live], ref[live])
    print("max rel err %.3e" % err)
    assert err <= TOL_F32
    assert np.all(out[~live] == 0.0)


def test_polar_decode_split_invariance_bf16(cuda, tqlib):
    outs = []
    for s in (1, 4, 16):
        out, ref = decode_case(cuda, tqlib, B=2, Hq=8, Hkv=2, ctx=[700, 513], bits_k=4, bits_v=4, seed=2,
                               num_splits=s, out_f32=False)
        assert max_rel_err(out, ref) <= TOL_BF16
        outs.append(out)
    assert max_rel_err(outs[0], outs[2]) <= TOL_BF16


def test_polar_append_then_decode_end_to_end(cuda, tqlib):
    """GPU append of bf16 K/V and GPU decode against the oracle's own encoding and exact
    attention of the same inputs (code mismatches in the edge band included)."""
    tq = tqlib
    B, Hq, Hkv, T = 3, 8, 2, 400
    mb = math.ceil(T / 16)
    bt, nb = workloads.shuffled_block_table(21, B, mb, num_blocks=B * mb + 2)
    layer = tq.Layer(nb, Hkv, kv_format="polar", bits_k=4, bits_v=3, seed=13, layer=4)
    kb, vb = workloads.heavy_tail_kv(8, B * T, Hkv, D)
    slots = workloads.prefill_slots(bt, T)
    layer.append(dev_bf16(cuda, kb), dev_bf16(cuda, vb), cuda.from_numpy(slots.astype(np.int64)).cuda())
    ctx = np.array([T, 1, 257], np.int32)
    qf = workloads.queries(5, B, Hq, D)
    out = layer.decode(dev_bf16(cuda, qf), cuda.from_numpy(bt).cuda(), cuda.from_numpy(ctx).cuda(),
                       sm_scale=1.0 / math.sqrt(D), out_dtype=cuda.float32).cpu().numpy()
    cuda.cuda.synchronize()
    assert tq.get_device_status() == 0
    pi = orot.hadamard_rotation_seeded(13, 4, D)
    kpool, vpool = oracle_pools(0, nb, Hkv, 4, 3, pi, oq.bf16_bits_to_f64(kb), oq.bf16_bits_to_f64(vb), slots)
    ref = opolar.decode_attention(oq.bf16_bits_to_f64(qf), kpool, vpool, pi, 4, 3, nb, Hkv, bt, ctx,
                                  1.0 / math.sqrt(D))
    err = max_rel_err(out, ref)
    print("end-to-end max rel err %.3e" % err)
    assert err <= TOL_BF16


def test_polar_decode_flags_bad_block(cuda, tqlib):
    tq = tqlib
    layer = tq.Layer(8, 1, kv_format="polar")
    bt = cuda.tensor([[0, 99]], dtype=cuda.int32).cuda()
    q = cuda.zeros((1, 4, D), dtype=cuda.float32).cuda()
    layer.decode(q, bt, cuda.tensor([20], dtype=cuda.int32).cuda(), sm_scale=0.1, out_dtype=cuda.float32)
    assert tq.get_device_status() & tq.TQ_DEV_BAD_BLOCK


def test_polar_full_size_sampled(cuda, tqlib):
    """The benchmark shape (16 sequences x 8192 tokens, 32 query / 8 KV heads, 4-bit
    angles): prefill append and decode on the GPU; three (sequence, KV head) units
    checked against the oracle's encoding and exact attention."""
    tq = tqlib
    B, Hq, Hkv, T = 16, 32, 8, 8192
    mb = T // 16
    bt, nb = workloads.shuffled_block_table(1234, B, mb)
    layer = tq.Layer(nb, Hkv, kv_format="polar", bits_k=4, bits_v=4, seed=17, layer=0)
    kb, vb = workloads.lognormal_channel_kv(77, B * T, Hkv, D)
    slots = workloads.prefill_slots(bt, T)
    layer.append(dev_bf16(cuda, kb), dev_bf16(cuda, vb), cuda.from_numpy(slots.astype(np.int64)).cuda())
    ctx = np.full(B, T, np.int32)
    qf = workloads.queries(99, B, Hq, D)
    sm = 1.0 / math.sqrt(D)
    out = layer.decode(dev_bf16(cuda, qf), cuda.from_numpy(bt).cuda(), cuda.from_numpy(ctx).cuda(), sm_scale=sm,
                       out_dtype=cuda.float32).cpu().numpy()
    assert tq.get_device_status() == 0
    pi = orot.hadamard_rotation_seeded(17, 0, D)
    kx = oq.bf16_bits_to_f64(kb).reshape(B, T, Hkv, D)
    vx = oq.bf16_bits_to_f64(vb).reshape(B, T, Hkv, D)
    qx = oq.bf16_bits_to_f64(qf)
    g = Hq // Hkv
    for b, kvh in ((0, 0), (7, 5), (15, 7)):
        kh = opolar.decode(*opolar.encode(kx[b, :, kvh], pi, 4), pi, 4)
        vh = opolar.decode(*opolar.encode(vx[b, :, kvh], pi, 4), pi, 4)
        for h in range(kvh * g, (kvh + 1) * g):
            s = sm * (kh @ qx[b, h])
            w = np.exp(s - s.max())
            ref = (w / w.sum()) @ vh
            assert max_rel_err(out[b, h][None], ref[None]) <= TOL_BF16


def test_polar_append_decode_fused_equals_separate_calls(cuda, tqlib):
    """tq_append_decode on a polar layer: the same pages and the same output as
    tq_quantize_append followed by tq_decode_attention."""
    tq = tqlib
    B, Hq, Hkv, T = 2, 8, 2, 150
    mb = math.ceil((T + 1) / 16)
    bt, nb = workloads.shuffled_block_table(31, B, mb, num_blocks=B * mb + 1)
    kb, vb = workloads.lognormal_channel_kv(33, B * T, Hkv, D)
    nk, nv = workloads.lognormal_channel_kv(34, B, Hkv, D)  # one new token per sequence
    slots = cuda.from_numpy(workloads.prefill_slots(bt, T).astype(np.int64)).cuda()
    new_slots = cuda.from_numpy(workloads.slot_mapping(bt, np.full((B, 1), T)).reshape(-1).astype(np.int64)).cuda()
    ctx = cuda.from_numpy(np.full(B, T + 1, np.int32)).cuda()
    q = dev_bf16(cuda, workloads.queries(35, B, Hq, D))
    btd = cuda.from_numpy(bt).cuda()
    outs, pools = [], []
    for fused in (False, True):
        layer = tq.Layer(nb, Hkv, kv_format="polar", bits_k=3, bits_v=4, seed=3, layer=1)
        layer.append(dev_bf16(cuda, kb), dev_bf16(cuda, vb), slots)
        if fused:
            out = layer.append_decode(dev_bf16(cuda, nk), dev_bf16(cuda, nv), new_slots, q, btd, ctx,
                                      out_dtype=cuda.float32)
        else:
            layer.append(dev_bf16(cuda, nk), dev_bf16(cuda, nv), new_slots)
            out = layer.decode(q, btd, ctx, out_dtype=cuda.float32)
        outs.append(out.cpu().numpy())
        pools.append((layer.k_cache.cpu().numpy(), layer.v_cache.cpu().numpy()))
    assert tq.get_device_status() == 0
    assert np.array_equal(pools[0][0], pools[1][0]) and np.array_equal(pools[0][1], pools[1][1])
    assert np.array_equal(outs[0], outs[1])
