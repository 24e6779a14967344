"""GPU decode and dequantize on caches the oracle quantized and packed itself.

The other decode tests compare the GPU with the oracle's attention over the
GPU's own packed cache.  Here the oracle encodes the inputs (its own rotation,
codebook, QJL projection and FP8 encoder, from the same seeds), packs the pages
and the bytes are uploaded into the layer's pools, so every oracle input is
computed on the CPU; the GPU's decode and dequantize of those pages must match
the oracle's within the usual tolerances.  The end-to-end test also encodes on
the GPU and compares with the oracle's own encoding of the same inputs (codes
may differ inside the tie band, hence the bf16 tolerance)."""
import math

import numpy as np
import pytest

import workloads
from oracle import attention as oa, codebook as ocb, fp8 as ofp8, pack as opack, qjl as oqjl
from oracle import quantize as oq, rotation as orot, rng as orng
from tests._gpu_util import D, max_rel_err

pytestmark = pytest.mark.gpu

TOL_F32 = 2e-3
TOL_BF16 = 5e-3


def write_packed(pool, slots, h, H, bits, idx, gamma, signs=None, rho=None):
    for t, s in enumerate(slots):
        if signs is None:
            opack.write_record(pool, int(s), h, H, D, bits, idx[t], gamma[t])
        else:
            opack.write_record(pool, int(s), h, H, D, bits, idx[t], gamma[t], signs[t], rho[t])


def oracle_layer_pools(nb, H, kx, vx, slots, *, bits_k, bits_v, pi, qjl_s=None, k8=False):
    """Host K/V pools written by the oracle, and the oracle's view of the layer."""
    cbv = ocb.codebook_fp32(D, bits_v)
    if k8:
        kpool = np.zeros(nb * H * ofp8.page_bytes(D), np.uint8)
        pages = kpool.reshape(nb, H, 16, D)
        for h in range(H):
            pages[slots // 16, h, slots % 16] = ofp8.encode(kx[:, h])
        cbk = (np.zeros(16), np.zeros(15))
    else:
        cbk = ocb.codebook_fp32(D, bits_k)
        kpool = np.zeros(nb * H * opack.page_bytes(D, bits_k, qjl_s is not None), np.uint8)
        for h in range(H):
            if qjl_s is None:
                idx, gamma, _ = oq.quantize(kx[:, h], pi, cbk[0], cbk[1])
                write_packed(kpool, slots, h, H, bits_k, idx, gamma)
            else:
                idx, gamma, signs, rho, _ = oqjl.residual_encode(kx[:, h], pi, cbk[0], cbk[1], qjl_s)
                write_packed(kpool, slots, h, H, bits_k, idx, gamma, signs, rho)
    vpool = np.zeros(nb * H * opack.page_bytes(D, bits_v), np.uint8)
    for h in range(H):
        idx, gamma, _ = oq.quantize(vx[:, h], pi, cbv[0], cbv[1])
        write_packed(vpool, slots, h, H, bits_v, idx, gamma)
    layer = oa.PackedLayer(pi, cbk[0], cbv[0], 8 if k8 else bits_k, bits_v, qjl_s)
    return kpool, vpool, layer


def upload(cuda, layer, kpool, vpool):
    assert layer.k_cache.numel() == kpool.size and layer.v_cache.numel() == vpool.size
    layer.k_cache.copy_(cuda.from_numpy(kpool).cuda())
    layer.v_cache.copy_(cuda.from_numpy(vpool).cuda())


def dev_bf16(cuda, bits):
    return cuda.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(cuda.bfloat16)


def run(cuda, tq, *, kv_format="packed", bits_k=4, bits_v=4, qjl=False, rot=orng.KIND_HADAMARD, B=3, Hq=8, Hkv=2,
        ctx=(300, 17, 129), q_f32=True, num_splits=0, seed=0):
    ctx = np.asarray(ctx, np.int32)
    mb = int(math.ceil(ctx.max() / 16))
    bt, nb = workloads.shuffled_block_table(seed + 1, B, mb, num_blocks=B * mb + 2)
    kb, vb = workloads.lognormal_channel_kv(seed + 2, B * mb * 16, Hkv, D)
    kx, vx = oq.bf16_bits_to_f64(kb), oq.bf16_bits_to_f64(vb)
    slots = workloads.prefill_slots(bt, mb * 16)
    k8 = kv_format == "k8v4"
    layer = tq.Layer(nb, Hkv, kv_format=kv_format, bits_k=bits_k, bits_v=bits_v, qjl=qjl, rot_kind=rot,
                     seed=seed + 5, layer=seed % 4, qjl_seed=seed + 9)
    pi = orot.rotation_seeded(rot, seed + 5, seed % 4, D)
    s = orot.qjl_matrix_seeded(seed + 9, D, D) if qjl else None
    kpool, vpool, ol = oracle_layer_pools(nb, Hkv, kx, vx, slots, bits_k=bits_k, bits_v=bits_v, pi=pi, qjl_s=s,
                                          k8=k8)
    upload(cuda, layer, kpool, vpool)
    qf = workloads.queries(seed + 3, B, Hq, D, dtype="f32" if q_f32 else "bf16")
    qd = cuda.from_numpy(qf).cuda() if q_f32 else dev_bf16(cuda, qf)
    sm = 1.0 / math.sqrt(D)
    out = layer.decode(qd, cuda.from_numpy(bt).cuda(), cuda.from_numpy(ctx).cuda(), sm_scale=sm,
                       out_dtype=cuda.float32, num_splits=num_splits).cpu().numpy()
    assert tq.get_device_status() == 0
    qx = qf.astype(np.float64) if q_f32 else oq.bf16_bits_to_f64(qf)
    if k8:
        ref = oa.decode_k8v4(qx, kpool, vpool, ol, nb, Hkv, bt, ctx, sm)
    else:
        ref = oa.decode_packed(qx, kpool, vpool, ol, nb, Hkv, bt, ctx, sm)
    live = ctx > 0
    return max_rel_err(out[live], ref[live]), layer, (kpool, vpool, ol, slots, kx, vx)


@pytest.mark.parametrize("case", [
    dict(bits_k=4, bits_v=4),
    dict(bits_k=3, bits_v=4, Hq=16, ctx=(250, 0, 96)),           # groups of 8, an empty sequence
    dict(bits_k=2, bits_v=2, Hq=2, num_splits=3),                 # g = 1
    dict(bits_k=4, bits_v=4, rot=orng.KIND_DENSE),                # dense rotation (query mat-vec pass)
    dict(bits_k=2, bits_v=4, qjl=True),                           # QJL keys
    dict(bits_k=3, bits_v=2, qjl=True),                           # LMDeploy layout
    dict(kv_format="k8v4", bits_k=8, bits_v=4),                   # FP8 keys
    dict(bits_k=4, bits_v=3, q_f32=False),                        # bf16 query
])
def test_decode_on_oracle_packed_pages(cuda, tqlib, case):
    err, _, _ = run(cuda, tqlib, seed=len(case), **case)
    tol = TOL_F32 if case.get("q_f32", True) else TOL_BF16
    print("max rel err %.3e" % err)
    assert err <= tol


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_dequantize_oracle_packed_pages(cuda, tqlib, bits):
    _, layer, (kpool, vpool, ol, slots, kx, vx) = run(cuda, tqlib, bits_k=bits, bits_v=bits, seed=20 + bits)
    sl = slots[::7].astype(np.int64)
    for which, pool, cb in ((0, kpool, ol.cb_k), (1, vpool, ol.cb_v)):
        out = layer.dequantize(which, cuda.from_numpy(sl).cuda(), out_dtype=cuda.float32).cpu().numpy()
        for h in range(layer.num_kv_heads):
            rec = [opack.read_record(pool, int(s), h, layer.num_kv_heads, D, bits) for s in sl]
            idx = np.array([r[0] for r in rec])
            gamma = np.array([r[1] for r in rec])
            ref = oq.dequantize(idx, gamma, ol.pi, cb)
            assert max_rel_err(out[:, h], ref) <= 1e-5


def test_end_to_end_against_the_oracles_own_encoding(cuda, tqlib):
    """GPU append of bf16 K/V + GPU decode vs the oracle's quantization of the same
    inputs and its exact attention (4-bit K/V, lognormal channels, ragged contexts)."""
    tq = tqlib
    B, Hq, Hkv = 3, 8, 2
    ctx = np.array([400, 1, 257], np.int32)
    mb = math.ceil(ctx.max() / 16)
    bt, nb = workloads.shuffled_block_table(41, B, mb, num_blocks=B * mb + 2)
    kb, vb = workloads.lognormal_channel_kv(42, B * mb * 16, Hkv, D)
    slots = workloads.prefill_slots(bt, mb * 16)
    layer = tq.Layer(nb, Hkv, bits_k=4, bits_v=4, seed=43, layer=1)
    layer.append(dev_bf16(cuda, kb), dev_bf16(cuda, vb), cuda.from_numpy(slots.astype(np.int64)).cuda())
    qf = workloads.queries(44, B, Hq, D)
    out = layer.decode(dev_bf16(cuda, qf), cuda.from_numpy(bt).cuda(), cuda.from_numpy(ctx).cuda(),
                       out_dtype=cuda.float32).cpu().numpy()
    assert tq.get_device_status() == 0
    pi = orot.rotation_seeded(orng.KIND_HADAMARD, 43, 1, D)
    kpool, vpool, ol = oracle_layer_pools(nb, Hkv, oq.bf16_bits_to_f64(kb), oq.bf16_bits_to_f64(vb), slots,
                                          bits_k=4, bits_v=4, pi=pi)
    ref = oa.decode_packed(oq.bf16_bits_to_f64(qf), kpool, vpool, ol, nb, Hkv, bt, ctx, 1.0 / math.sqrt(D))
    err = max_rel_err(out, ref)
    print("end-to-end max rel err %.3e" % err)
    assert err <= TOL_BF16
