"""GPU parity of the k8v4 layer format (FP8 E4M3 keys, TurboQuant values) against
the oracle: key bytes bit-exact with the oracle's FP8 encoding, values within the
tie band, decode attention within the decode tolerances."""
import math

import numpy as np
import pytest

import workloads
from oracle import attention as oa, codebook as ocb, fp8, quantize as oq
from tests._gpu_util import D, max_rel_err, oracle_pi, page_fields, slot_fields, tie_band_ok

pytestmark = pytest.mark.gpu

TOL_F32 = 2e-3
TOL_BF16 = 5e-3


def k8v4_oracle_layer(layer):
    cbv = ocb.codebook_fp32(D, layer.bits_v)[0]
    return oa.PackedLayer(oracle_pi(layer), np.zeros(16), cbv, 8, layer.bits_v)


def key_records(layer, pool_host):
    """uint8 [num_blocks, H_kv, 16, d] view of an FP8 key pool."""
    return np.asarray(pool_host, np.uint8).reshape(layer.num_blocks, layer.num_kv_heads, 16, D)


def to_dev(cuda, arr, bf16):
    if bf16:
        return cuda.from_numpy(np.ascontiguousarray(arr).view(np.int16)).cuda().view(cuda.bfloat16)
    return cuda.from_numpy(np.ascontiguousarray(arr)).cuda()


def make_slots(cuda, n, num_blocks, seed, skip_every=0):
    perm = np.random.default_rng(seed).permutation(num_blocks * 16)[:n].astype(np.int64)
    if skip_every:
        perm[::skip_every] = -1
    return perm, cuda.from_numpy(perm).cuda()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_k8v4_append_keys_bit_exact(cuda, tqlib, dtype):
    """Key bytes equal the oracle's E4M3 encoding of the inputs (saturation at 448,
    subnormals, signed zeros included); values match the oracle within the tie band;
    skipped slots keep their fill."""
    tq = tqlib
    H, nb, n = 2, 30, 401
    layer = tq.Layer(nb, H, kv_format="k8v4", bits_v=4, seed=6, layer=3, fill=0x5A)
    g = np.random.default_rng(70)
    x = g.standard_normal((n, H, D)).astype(np.float32) * np.float32(40.0)
    x[:40] *= np.float32(30.0)                        # beyond 448: saturates
    x[40:80] *= np.float32(1e-4)                      # subnormal range
    x[80, 0, :4] = np.array([0.0, -0.0, 448.0, -464.0], np.float32)
    v = g.standard_normal((n, H, D)).astype(np.float32)
    if dtype == "bf16":
        xb, vb = workloads.bf16_bits(x), workloads.bf16_bits(v)
        kx, vx = oq.bf16_bits_to_f64(xb), oq.bf16_bits_to_f64(vb)
        kt, vt = to_dev(cuda, xb, True), to_dev(cuda, vb, True)
    else:
        kx, vx = x.astype(np.float64), v.astype(np.float64)
        kt, vt = to_dev(cuda, x, False), to_dev(cuda, v, False)
    slots, slots_d = make_slots(cuda, n, nb, 71, skip_every=13)
    layer.append(kt, vt, slots_d)
    assert tq.get_device_status() == 0
    keep = slots >= 0
    recs = key_records(layer, layer.k_cache.cpu().numpy())
    got = recs[slots[keep] // 16, :, slots[keep] % 16]  # [n_keep, H, d]
    assert np.array_equal(got, fp8.encode(kx[keep]))
    written = np.zeros(nb * 16, bool)
    written[slots[keep]] = True
    assert np.all(recs.transpose(0, 2, 1, 3).reshape(nb * 16, H, D)[~written] == 0x5A)
    pi = oracle_pi(layer)
    c32, b32 = ocb.codebook_fp32(D, 4)
    fields = page_fields(layer, 1, layer.v_cache.cpu().numpy())
    for h in range(H):
        idx, gamma, y = oq.quantize(vx[keep, h], pi, c32, b32)
        codes, g_gpu = slot_fields(fields, slots[keep], h)
        ok, _ = tie_band_ok(y, codes, idx, b32, 1e-5)
        assert ok
        same = np.all(codes == idx, axis=-1)
        assert np.all(np.abs(g_gpu[same] - gamma[same]) <= 1e-6 * np.abs(gamma[same]) + 1e-30)


def run_k8v4(cuda, tq, *, B, Hq, Hkv, ctx, rot, bits_v=4, q_f32=False, num_splits=0, seed=0, scale=8.0):
    ctx = np.asarray(ctx, np.int32)
    mb = int(max(1, math.ceil(ctx.max() / 16)))
    bt, nb = workloads.shuffled_block_table(seed + 1, B, mb, num_blocks=B * mb + 2)
    tmax = mb * 16
    kb, vb = workloads.lognormal_channel_kv(seed, B * tmax, Hkv, D)
    kb = workloads.bf16_bits(workloads.bf16_to_f32(kb) * np.float32(scale)).reshape(B, tmax, Hkv, D)
    vb = vb.reshape(B, tmax, Hkv, D)
    layer = tq.Layer(nb, Hkv, kv_format="k8v4", bits_v=bits_v, rot_kind=rot, seed=seed + 2, layer=seed % 7)
    slots = np.concatenate([workloads.slot_mapping(bt[b:b + 1], np.arange(ctx[b])[None, :])[0] for b in range(B)])
    k = np.concatenate([kb[b, : ctx[b]] for b in range(B)])
    v = np.concatenate([vb[b, : ctx[b]] for b in range(B)])
    layer.append(to_dev(cuda, k, True), to_dev(cuda, v, True), cuda.from_numpy(slots.astype(np.int64)).cuda())
    qf = workloads.queries(seed + 9, B, Hq, D, dtype="f32" if q_f32 else "bf16")
    qd = to_dev(cuda, qf, not q_f32)
    sm = 1.0 / math.sqrt(D)
    out = layer.decode(qd, cuda.from_numpy(bt).cuda(), cuda.from_numpy(ctx).cuda(), sm_scale=sm,
                       out_dtype=cuda.float32, num_splits=num_splits)
    cuda.cuda.synchronize()
    assert tq.get_device_status() == 0
    qx = qf.astype(np.float64) if q_f32 else oq.bf16_bits_to_f64(qf)
    ref = oa.decode_k8v4(qx, layer.k_cache.cpu().numpy(), layer.v_cache.cpu().numpy(), k8v4_oracle_layer(layer), nb,
                         Hkv, bt, ctx, sm)
    return out.cpu().numpy(), ref, layer, (qd, bt, ctx)


@pytest.mark.parametrize("hq,hkv,rot", [(8, 2, 1), (16, 2, 1), (8, 2, 2)])
def test_k8v4_decode_matches_oracle(cuda, tqlib, hq, hkv, rot):
    """Groups of 4 and 8 query heads, Hadamard and dense value rotations, ragged
    contexts (one token, a partial block, several splits)."""
    out, ref, _, _ = run_k8v4(cuda, tqlib, B=3, Hq=hq, Hkv=hkv, ctx=[700, 23, 1], rot=rot, seed=hq + rot)
    err = max_rel_err(out.reshape(-1, D), ref.reshape(-1, D))
    print("k8v4 max rel err %.3e" % err)
    assert err <= TOL_BF16


def test_k8v4_fp32_query_and_split_invariance(cuda, tqlib):
    out1, ref, layer, (qd, bt, ctx) = run_k8v4(cuda, tqlib, B=2, Hq=8, Hkv=2, ctx=[513, 300], rot=1, q_f32=True,
                                              num_splits=1, seed=3)
    assert max_rel_err(out1.reshape(-1, D), ref.reshape(-1, D)) <= TOL_F32
    out7 = layer.decode(qd, cuda.from_numpy(bt).cuda(), cuda.from_numpy(ctx).cuda(), out_dtype=cuda.float32,
                        num_splits=7).cpu().numpy()
    assert max_rel_err(out7.reshape(-1, D), out1.reshape(-1, D)) <= 1e-5


def test_k8v4_append_decode_and_dequantize(cuda, tqlib):
    """The fused append + decode equals the two calls; tq_dequantize of the keys gives
    the stored FP8 values exactly."""
    tq = tqlib
    B, Hq, Hkv, T = 2, 8, 2, 96
    bt, nb = workloads.shuffled_block_table(4, B, T // 16, num_blocks=B * T // 16 + 1)
    kw = dict(kv_format="k8v4", bits_v=3, seed=1, layer=2)
    la, lb = tq.Layer(nb, Hkv, **kw), tq.Layer(nb, Hkv, **kw)
    kb, vb = workloads.scaled_gaussian_kv(5, B * T, Hkv, D, scale=20.0)
    kb, vb = kb.reshape(B, T, Hkv, D), vb.reshape(B, T, Hkv, D)
    pos = np.array([50, 71], np.int32)
    slots = workloads.slot_mapping(bt, pos[:, None])[:, 0].astype(np.int64)
    knew, vnew = to_dev(cuda, kb[np.arange(B), pos], True), to_dev(cuda, vb[np.arange(B), pos], True)
    slots_d = cuda.from_numpy(slots).cuda()
    q = to_dev(cuda, workloads.queries(3, B, Hq, D), True)
    ctx_d = cuda.from_numpy(pos + 1).cuda()
    bt_d = cuda.from_numpy(bt).cuda()
    out_a = la.append_decode(knew, vnew, slots_d, q, bt_d, ctx_d, out_dtype=cuda.float32)
    lb.append(knew, vnew, slots_d)
    out_b = lb.decode(q, bt_d, ctx_d, out_dtype=cuda.float32)
    cuda.cuda.synchronize()
    assert tq.get_device_status() == 0
    assert np.array_equal(out_a.cpu().numpy(), out_b.cpu().numpy())
    assert np.array_equal(la.k_cache.cpu().numpy(), lb.k_cache.cpu().numpy())
    assert np.array_equal(la.v_cache.cpu().numpy(), lb.v_cache.cpu().numpy())
    kd = la.dequantize(0, slots_d).cpu().numpy()
    recs = key_records(la, la.k_cache.cpu().numpy())
    assert np.array_equal(kd.astype(np.float64), fp8.decode(recs[slots // 16, :, slots % 16]))


def test_k8v4_llama8b_shape_full_size_sampled(cuda, tqlib):
    """Batch 16, 32/8 heads, context 8192 with lognormal channels and a shuffled table,
    k8v4 with 4-bit values; sampled (sequence, KV head) pairs of the full-size run."""
    tq, torch = tqlib, cuda
    B, Hq, Hkv, T = 16, 32, 8, 8192
    bt, nb = workloads.shuffled_block_table(61, B, T // 16 + 1)
    layer = tq.Layer(nb, Hkv, kv_format="k8v4", bits_v=4, seed=0, layer=5)
    gen = torch.Generator(device="cuda").manual_seed(62)
    sk = torch.exp(torch.randn(Hkv, D, generator=gen, device="cuda"))
    sv = torch.exp(torch.randn(Hkv, D, generator=gen, device="cuda"))
    k = (torch.randn(B * T, Hkv, D, generator=gen, device="cuda") * sk).to(torch.bfloat16)
    v = (torch.randn(B * T, Hkv, D, generator=gen, device="cuda") * sv).to(torch.bfloat16)
    layer.append(k, v, torch.from_numpy(workloads.prefill_slots(bt, T)).cuda())
    del k, v
    ctx = np.full(B, T, np.int32)
    q = torch.randn(B, Hq, D, generator=gen, device="cuda").to(torch.bfloat16)
    out = layer.decode(q, torch.from_numpy(bt).cuda(), torch.from_numpy(ctx).cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tq.get_device_status() == 0
    kp, vp = layer.k_cache.cpu().numpy(), layer.v_cache.cpu().numpy()
    ol = k8v4_oracle_layer(layer)
    qx = q.float().cpu().numpy().astype(np.float64)
    o = out.cpu().numpy()
    errs = []
    for b, kvh in ((0, 0), (9, 4), (15, 7)):
        kk, vv = oa.gather_k8v4(kp, vp, ol, nb, Hkv, D, bt[b], T, kvh)
        for h in range(kvh * 4, kvh * 4 + 4):
            errs.append(max_rel_err(o[b, h][None], oa.softmax_attention(qx[b, h], kk, vv, 1 / math.sqrt(D))[None]))
    print("k8v4 sampled max rel err %.3e" % max(errs))
    assert max(errs) <= TOL_BF16
