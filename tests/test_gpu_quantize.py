"""GPU parity of quantize-on-append, the quantizer alone, bf16 append and
dequantize against the oracle (all through the C ABI via the binding)."""
import numpy as np
import pytest

import workloads
from oracle import codebook as ocb, quantize as oq, qjl as oqjl, rotation as orot
from tests._gpu_util import D, oracle_pi, page_fields, slot_fields, tie_band_ok

pytestmark = pytest.mark.gpu


def make_slots(cuda, n, num_blocks, seed, skip_every=0):
    perm = np.random.default_rng(seed).permutation(num_blocks * 16)[:n].astype(np.int64)
    if skip_every:
        perm[::skip_every] = -1
    return perm, cuda.from_numpy(perm).cuda()


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_quantizer_bit_exact_given_rotated_coordinates(cuda, tqlib, bits):
    tq = tqlib
    H, nb, n = 3, 40, 301  # 903 vectors: several CTA tiles and a ragged tail
    layer = tq.Layer(nb, H, bits_k=bits, bits_v=bits, fill=0xA5)
    c32, b32 = ocb.codebook_fp32(D, bits)
    g = np.random.default_rng(bits)
    x = g.standard_normal((n, H, D))
    y = (x / np.linalg.norm(x, axis=-1, keepdims=True)).astype(np.float32)
    # plant exact boundary values, their neighbours and signed zeros
    flat = y.reshape(-1)
    k = len(b32)
    flat[: 3 * k] = np.concatenate([b32, np.nextafter(b32, np.float32(-1)), np.nextafter(b32, np.float32(1))])
    flat[3 * k: 3 * k + 4] = np.array([0.0, -0.0, 1e-30, -1e-30], np.float32)
    norms = (g.random((n, H)) * 10 + 0.1).astype(np.float32)
    norms[5, 1] = 0.0
    slots, slots_d = make_slots(cuda, n, nb, 7, skip_every=17)
    layer.quantize_rotated(0, cuda.from_numpy(y).cuda(), cuda.from_numpy(norms).cuda(), slots_d)
    cuda.cuda.synchronize()
    kp = layer.k_cache.cpu().numpy()
    fields = page_fields(layer, 0, kp)
    expect = oq.codes_from_y(y, b32)
    for h in range(H):
        keep = slots >= 0
        codes, gamma = slot_fields(fields, slots[keep], h)
        assert np.array_equal(codes, expect[keep, h])
        cn = np.sqrt(np.sum(c32.astype(np.float64)[expect[keep, h]] ** 2, axis=-1))
        ref = norms[keep, h].astype(np.float64) / cn
        assert np.all(np.abs(gamma - ref) <= 1e-6 * np.abs(ref))
    # pages of skipped slots keep their 0xA5 fill
    skipped = slots[slots < 0]
    assert skipped.size > 0
    written = np.zeros(nb * 16, bool)
    written[slots[slots >= 0]] = True
    rec = opack_record_view(kp, nb, H, bits)
    assert np.all(rec[~written.reshape(nb, 16)] == 0xA5)


def planted_coordinates(b32):
    """Rotated coordinates that sit on the quantizer's decision points: every
    boundary and its fp32 neighbours, the edges (i - 64) / 63 of the bulk
    kernels' 127 lookup cells and their neighbours, signed zeros, tiny values
    and the ends of [-1, 1] (with the first value past them)."""
    f32 = np.float32
    b32 = np.asarray(b32, f32)
    edges = ((np.arange(1, 128) - 64) / 63.0).astype(f32)
    pts = [b32, np.nextafter(b32, f32(-2)), np.nextafter(b32, f32(2)),
           edges, np.nextafter(edges, f32(-2)), np.nextafter(edges, f32(2)),
           np.array([0.0, -0.0, 1e-30, -1e-30, 1e-45, -1e-45, 1.0, -1.0], f32),
           np.array([np.nextafter(f32(1), f32(2)), np.nextafter(f32(-1), f32(-2))], f32)]
    return np.concatenate(pts).astype(f32)


@pytest.mark.parametrize("kind", ["hadamard_bulk", "dense"])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_bulk_quantizer_bit_exact_given_rotated_coordinates(cuda, tqlib, bits, kind):
    """The quantizer of the two bulk append kernels (the staged FWHT kernel for
    Hadamard appends of >= 24,576 vectors, the tensor-core kernel for dense
    layers) fed the oracle's y: codes equal the oracle's boundary count exactly,
    including coordinates planted on every boundary, its fp32 neighbours and
    the edges of the kernels' lookup cells."""
    tq = tqlib
    if kind == "hadamard_bulk":
        H, nb, n = 8, 200, 3079  # 24,632 vectors: the bulk path, with a ragged last tile
        layer = tq.Layer(nb, H, bits_k=bits, bits_v=bits, fill=0xA5)
    else:
        H, nb, n = 3, 40, 301
        layer = tq.Layer(nb, H, bits_k=bits, bits_v=bits, fill=0xA5, rot_kind=tq.TQ_ROT_DENSE, seed=2, layer=3)
    c32, b32 = ocb.codebook_fp32(D, bits)
    g = np.random.default_rng(100 + bits)
    x = g.standard_normal((n, H, D))
    y = (x / np.linalg.norm(x, axis=-1, keepdims=True)).astype(np.float32)
    flat = y.reshape(-1)
    pts = planted_coordinates(b32)
    # each planted value at several coordinates of different vectors (every position mod 128 is hit)
    for r in range(4):
        idx = (np.arange(pts.size) * 131 + r * 977) % flat.size
        flat[idx] = pts
    norms = (g.random((n, H)) * 10 + 0.1).astype(np.float32)
    norms[5, 1] = 0.0
    slots, slots_d = make_slots(cuda, n, nb, 11, skip_every=17)
    layer.quantize_rotated(1, cuda.from_numpy(y).cuda(), cuda.from_numpy(norms).cuda(), slots_d)
    cuda.cuda.synchronize()
    assert tq.get_device_status() == 0
    vp = layer.v_cache.cpu().numpy()
    fields = page_fields(layer, 1, vp)
    expect = oq.codes_from_y(y, b32)
    keep = slots >= 0
    for h in range(H):
        codes, gamma = slot_fields(fields, slots[keep], h)
        assert np.array_equal(codes, expect[keep, h]), (h, int(np.sum(codes != expect[keep, h])))
        cn = np.sqrt(np.sum(c32.astype(np.float64)[expect[keep, h]] ** 2, axis=-1))
        ref = norms[keep, h].astype(np.float64) / cn
        assert np.all(np.abs(gamma - ref) <= 1e-6 * np.abs(ref))
    written = np.zeros(nb * 16, bool)
    written[slots[keep]] = True
    rec = opack_record_view(vp, nb, H, bits)
    assert np.all(rec[~written.reshape(nb, 16)] == 0xA5)


def opack_record_view(pool, nb, H, bits):
    """uint8 [nb, 16, H, record+4] view of code records and gammas (for fill checks)."""
    from oracle import pack as opack
    pb = opack.page_bytes(D, bits)
    pages = pool.reshape(nb, H, pb)
    rb = opack.record_bytes(D, bits)
    codes = pages[:, :, : 16 * rb].reshape(nb, H, 16, rb)
    gam = pages[:, :, 16 * rb: 16 * rb + 64].reshape(nb, H, 16, 4)
    return np.concatenate([codes, gam], axis=-1).transpose(0, 2, 1, 3)


@pytest.mark.parametrize("bits,dtype", [(4, "f32"), (3, "bf16"), (2, "bf16"), (4, "bf16")])
def test_append_hadamard_matches_oracle_within_tie_band(cuda, tqlib, bits, dtype):
    tq = tqlib
    H, nb, n = 2, 24, 257
    layer = tq.Layer(nb, H, bits_k=bits, bits_v=bits, seed=3, layer=1)
    if dtype == "f32":
        k, v, _, _ = workloads.tiny_kv(seed=1, n_tokens=n, d=D)
        k = np.repeat(k, H, axis=1) * np.array([1.0, 0.01], np.float32)[None, :, None]
        v = np.repeat(v, H, axis=1)
        kx, vx = k.astype(np.float64), v.astype(np.float64)
        kt, vt = cuda.from_numpy(k).cuda(), cuda.from_numpy(v).cuda()
    else:
        kb, vb = workloads.lognormal_channel_kv(2, n, H, D)
        kx, vx = oq.bf16_bits_to_f64(kb), oq.bf16_bits_to_f64(vb)
        kt = cuda.from_numpy(kb.view(np.int16)).cuda().view(cuda.bfloat16)
        vt = cuda.from_numpy(vb.view(np.int16)).cuda().view(cuda.bfloat16)
    slots, slots_d = make_slots(cuda, n, nb, 11)
    layer.append(kt, vt, slots_d)
    assert tq.get_device_status() == 0
    pi = orot.hadamard_rotation_seeded(3, 1, D)
    c32, b32 = ocb.codebook_fp32(D, bits)
    kp, vp = layer.k_cache.cpu().numpy(), layer.v_cache.cpu().numpy()
    total_mism = 0.0
    for which, x, pool in ((0, kx, kp), (1, vx, vp)):
        fields = page_fields(layer, which, pool)
        for h in range(H):
            idx, gamma, y = oq.quantize(x[:, h], pi, c32, b32)
            codes, g_gpu = slot_fields(fields, slots, h)
            ok, rate = tie_band_ok(y, codes, idx, b32, 1e-5)
            assert ok, "code mismatch outside the tie band"
            total_mism += rate
            same = np.all(codes == idx, axis=-1)
            assert np.all(np.abs(g_gpu[same] - gamma[same]) <= 1e-6 * np.abs(gamma[same]) + 1e-30)
    print("tie-band mismatch rate (mean over K/V heads): %.2e" % (total_mism / (2 * H)))


def test_append_zero_vector_and_bad_slot(cuda, tqlib):
    tq = tqlib
    layer = tq.Layer(4, 1)
    x = np.zeros((2, 1, D), np.float32)
    x[1, 0, 3] = 2.0
    slots = cuda.tensor([5, 4 * 16 + 3], dtype=cuda.int64).cuda()  # second slot is out of range
    layer.append(cuda.from_numpy(x).cuda(), None, slots)
    assert tq.get_device_status() & tq.TQ_DEV_BAD_SLOT
    assert tq.get_device_status() == 0  # cleared by the read
    fields = page_fields(layer, 0, layer.k_cache.cpu().numpy())
    codes, gamma = slot_fields(fields, [5], 0)
    assert np.all(codes == 8) and gamma[0] == 0.0


def _bf16_dev(cuda, bits):
    return cuda.from_numpy(bits.view(np.int16)).cuda().view(cuda.bfloat16)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_append_bf16_many_tiles_per_warp(cuda, tqlib, bits):
    """8199 tokens x 8 heads of bf16 K and V in one paired launch (2 x 65592 vectors,
    a ragged last tile): large appends take the staged kernel, every warp of which
    refills its stage several times (the barrier phase flips from tile to tile)."""
    tq = tqlib
    H, n = 8, 8199
    nb = n // 16 + 3
    layer = tq.Layer(nb, H, bits_k=bits, bits_v=bits, seed=7, layer=3, fill=0xA5)
    kb, vb = workloads.lognormal_channel_kv(12, n, H, D)
    slots, slots_d = make_slots(cuda, n, nb, 13, skip_every=29)
    layer.append(_bf16_dev(cuda, kb), _bf16_dev(cuda, vb), slots_d)
    assert tq.get_device_status() == 0
    pi = orot.hadamard_rotation_seeded(7, 3, D)
    c32, b32 = ocb.codebook_fp32(D, bits)
    keep = slots >= 0
    written = np.zeros(nb * 16, bool)
    written[slots[keep]] = True
    for which, xb, pool in ((0, kb, layer.k_cache), (1, vb, layer.v_cache)):
        host = pool.cpu().numpy()
        fields = page_fields(layer, which, host)
        x = oq.bf16_bits_to_f64(xb)
        for h in range(H):
            idx, gamma, y = oq.quantize(x[keep, h], pi, c32, b32)
            codes, g_gpu = slot_fields(fields, slots[keep], h)
            ok, _ = tie_band_ok(y, codes, idx, b32, 1e-5)
            assert ok, "code mismatch outside the tie band"
            same = np.all(codes == idx, axis=-1)
            assert same.mean() > 0.99
            assert np.all(np.abs(g_gpu[same] - gamma[same]) <= 1e-6 * np.abs(gamma[same]) + 1e-30)
        rec = opack_record_view(host, nb, H, bits)
        assert np.all(rec[~written.reshape(nb, 16)] == 0xA5)


def test_append_bf16_keys_only_staged(cuda, tqlib):
    """A keys-only append of 4100 tokens x 8 heads (32800 vectors, one tensor per launch)."""
    tq = tqlib
    H, n = 8, 4100
    nb = n // 16 + 2
    layer = tq.Layer(nb, H, bits_k=4, bits_v=3, seed=2, layer=5, fill=0x3C)
    kb, _ = workloads.heavy_tail_kv(21, n, H, D)
    slots, slots_d = make_slots(cuda, n, nb, 17)
    layer.append(_bf16_dev(cuda, kb), None, slots_d)
    assert tq.get_device_status() == 0
    pi = orot.hadamard_rotation_seeded(2, 5, D)
    c32, b32 = ocb.codebook_fp32(D, 4)
    fields = page_fields(layer, 0, layer.k_cache.cpu().numpy())
    x = oq.bf16_bits_to_f64(kb)
    for h in range(H):
        idx, gamma, y = oq.quantize(x[:, h], pi, c32, b32)
        codes, g_gpu = slot_fields(fields, slots, h)
        ok, _ = tie_band_ok(y, codes, idx, b32, 1e-5)
        assert ok
        same = np.all(codes == idx, axis=-1)
        assert np.all(np.abs(g_gpu[same] - gamma[same]) <= 1e-6 * np.abs(gamma[same]) + 1e-30)
    assert np.all(layer.v_cache.cpu().numpy() == 0x3C)  # values untouched


def test_append_misaligned_input_rejected(cuda, tqlib):
    """k/v must be 16-byte aligned (include/tq.h): a bf16 input 2 bytes past a boundary is
    refused before anything is launched, and the cache is left as it was."""
    tq = tqlib
    H, nb, n = 2, 4, 9
    layer = tq.Layer(nb, H, fill=0x5A)
    kb, _ = workloads.lognormal_channel_kv(5, n, H, D)
    big = cuda.from_numpy(np.concatenate([np.zeros(1, np.int16), kb.view(np.int16).reshape(-1)])).cuda()
    kt = big[1:].view(n, H, D).view(cuda.bfloat16)
    assert kt.data_ptr() % 16 == 2
    slots = cuda.arange(n, dtype=cuda.int64).cuda()
    before = tq.launch_count()
    with pytest.raises(tq.TQError, match="16-byte aligned"):
        layer.append(kt, None, slots)
    assert tq.launch_count() == before
    assert np.all(layer.k_cache.cpu().numpy() == 0x5A)


def test_append_bf16_zero_vector_and_bad_slot(cuda, tqlib):
    tq = tqlib
    layer = tq.Layer(4, 1)
    x = np.zeros((2, 1, D), np.float32)
    x[1, 0, 3] = 2.0
    slots = cuda.tensor([5, 4 * 16 + 3], dtype=cuda.int64).cuda()  # second slot is out of range
    layer.append(_bf16_dev(cuda, workloads.bf16_bits(x)), None, slots)
    assert tq.get_device_status() & tq.TQ_DEV_BAD_SLOT
    assert tq.get_device_status() == 0
    fields = page_fields(layer, 0, layer.k_cache.cpu().numpy())
    codes, gamma = slot_fields(fields, [5], 0)
    assert np.all(codes == 8) and gamma[0] == 0.0


def test_dense_rotation_append_matches_oracle(cuda, tqlib):
    tq = tqlib
    H, nb, n = 2, 12, 150
    layer = tq.Layer(nb, H, rot_kind=tq.TQ_ROT_DENSE, seed=5, layer=2)
    kb, vb = workloads.scaled_gaussian_kv(4, n, H, D, scale=2.5)
    kt = cuda.from_numpy(kb.view(np.int16)).cuda().view(cuda.bfloat16)
    vt = cuda.from_numpy(vb.view(np.int16)).cuda().view(cuda.bfloat16)
    slots, slots_d = make_slots(cuda, n, nb, 3)
    layer.append(kt, vt, slots_d)
    pi = orot.dense_rotation_seeded(5, 2, D)
    c32, b32 = ocb.codebook_fp32(D, 4)
    for which, xb, pool in ((0, kb, layer.k_cache), (1, vb, layer.v_cache)):
        fields = page_fields(layer, which, pool.cpu().numpy())
        for h in range(H):
            idx, gamma, y = oq.quantize(oq.bf16_bits_to_f64(xb)[:, h], pi, c32, b32)
            codes, g_gpu = slot_fields(fields, slots, h)
            ok, rate = tie_band_ok(y, codes, idx, b32, 1e-5)
            assert ok
            same = np.all(codes == idx, axis=-1)
            assert np.all(np.abs(g_gpu[same] - gamma[same]) <= 2e-6 * gamma[same])


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_dense_rotation_append_tensor_cores_many_tiles(cuda, tqlib, bits):
    """bf16 appends through a dense Pi run as a tensor-core GEMM over tiles of 128
    vectors: 8199 tokens x 8 heads of K and V (2 x 65592 vectors, a ragged last
    tile, several tiles per CTA so the ring and the accumulators are reused)."""
    tq = tqlib
    H, n = 8, 8199
    nb = n // 16 + 3
    layer = tq.Layer(nb, H, bits_k=bits, bits_v=bits, rot_kind=tq.TQ_ROT_DENSE, seed=8, layer=7, fill=0x69)
    kb, vb = workloads.lognormal_channel_kv(31, n, H, D)
    slots, slots_d = make_slots(cuda, n, nb, 19, skip_every=37)
    layer.append(_bf16_dev(cuda, kb), _bf16_dev(cuda, vb), slots_d)
    assert tq.get_device_status() == 0
    pi = orot.dense_rotation_seeded(8, 7, D)
    c32, b32 = ocb.codebook_fp32(D, bits)
    keep = slots >= 0
    written = np.zeros(nb * 16, bool)
    written[slots[keep]] = True
    rates = []
    for which, xb, pool in ((0, kb, layer.k_cache), (1, vb, layer.v_cache)):
        host = pool.cpu().numpy()
        fields = page_fields(layer, which, host)
        x = oq.bf16_bits_to_f64(xb)
        for h in range(H):
            idx, gamma, y = oq.quantize(x[keep, h], pi, c32, b32)
            codes, g_gpu = slot_fields(fields, slots[keep], h)
            ok, rate = tie_band_ok(y, codes, idx, b32, 1e-5)
            assert ok, "code mismatch outside the tie band"
            rates.append(rate)
            same = np.all(codes == idx, axis=-1)
            assert same.mean() > 0.99
            assert np.all(np.abs(g_gpu[same] - gamma[same]) <= 2e-6 * gamma[same])
        rec = opack_record_view(host, nb, H, bits)
        assert np.all(rec[~written.reshape(nb, 16)] == 0x69)
    print("dense tensor-core append: tie-band mismatch rate %.2e" % np.mean(rates))


def test_dense_rotation_append_f32_input(cuda, tqlib):
    """fp32 inputs through a dense Pi (the CUDA-core mat-vec kernel)."""
    tq = tqlib
    H, nb, n = 2, 10, 140
    layer = tq.Layer(nb, H, rot_kind=tq.TQ_ROT_DENSE, seed=6, layer=1)
    x = np.random.default_rng(40).standard_normal((n, H, D)).astype(np.float32)
    slots, slots_d = make_slots(cuda, n, nb, 23)
    layer.append(cuda.from_numpy(x).cuda(), None, slots_d)
    assert tq.get_device_status() == 0
    pi = orot.dense_rotation_seeded(6, 1, D)
    c32, b32 = ocb.codebook_fp32(D, 4)
    fields = page_fields(layer, 0, layer.k_cache.cpu().numpy())
    for h in range(H):
        idx, gamma, y = oq.quantize(x[:, h].astype(np.float64), pi, c32, b32)
        codes, g_gpu = slot_fields(fields, slots, h)
        ok, _ = tie_band_ok(y, codes, idx, b32, 1e-5)
        assert ok
        same = np.all(codes == idx, axis=-1)
        assert np.all(np.abs(g_gpu[same] - gamma[same]) <= 2e-6 * gamma[same])


def test_qjl_residual_matches_oracle(cuda, tqlib):
    tq = tqlib
    H, nb, n = 2, 10, 130
    layer = tq.Layer(nb, H, bits_k=2, bits_v=4, qjl=True, seed=1, qjl_seed=9)
    kb, vb = workloads.scaled_gaussian_kv(6, n, H, D)
    kt = cuda.from_numpy(kb.view(np.int16)).cuda().view(cuda.bfloat16)
    slots, slots_d = make_slots(cuda, n, nb, 5)
    layer.append(kt, None, slots_d)
    pi = orot.hadamard_rotation_seeded(1, 0, D)
    s = orot.qjl_matrix_seeded(9, D, D)
    c32, b32 = ocb.codebook_fp32(D, 2)
    fields = page_fields(layer, 0, layer.k_cache.cpu().numpy())
    for h in range(H):
        x = oq.bf16_bits_to_f64(kb)[:, h]
        idx, gamma, signs, rho, r = oqjl.residual_encode(x, pi, c32, b32, s)
        codes, g_gpu, s_gpu, rho_gpu = slot_fields(fields, slots, h)
        same = np.all(codes == idx, axis=-1)
        assert same.mean() > 0.95
        # sign bits: mismatches only where |S r| is within rounding of 0
        z = r[same] @ s.T
        mism = s_gpu[same] != signs[same]
        scale = np.linalg.norm(s, axis=1)[None, :] * rho[same][:, None]
        assert np.all(np.abs(z[mism]) <= 1e-5 * scale[mism])
        assert np.all(np.abs(rho_gpu[same] - rho[same]) <= 1e-5 * rho[same] + 1e-6)


def test_bf16_layer_append_and_dequantize(cuda, tqlib):
    tq = tqlib
    H, nb, n = 2, 5, 37
    layer = tq.Layer(nb, H, kv_format="bf16")
    x = np.random.default_rng(0).standard_normal((n, H, D)).astype(np.float32)
    slots, slots_d = make_slots(cuda, n, nb, 2)
    layer.append(cuda.from_numpy(x).cuda(), cuda.from_numpy(x).cuda(), slots_d)
    back = layer.dequantize(0, slots_d).cpu().numpy()
    expect = workloads.bf16_to_f32(workloads.bf16_bits(x))
    assert np.array_equal(back, expect)


@pytest.mark.parametrize("rot", ["hadamard", "dense"])
def test_dequantize_matches_oracle(cuda, tqlib, rot):
    tq = tqlib
    H, nb, n = 2, 8, 90
    kind = tq.TQ_ROT_HADAMARD if rot == "hadamard" else tq.TQ_ROT_DENSE
    layer = tq.Layer(nb, H, bits_k=3, bits_v=4, rot_kind=kind, seed=2, layer=4)
    kb, vb = workloads.scaled_gaussian_kv(8, n, H, D)
    kt = cuda.from_numpy(kb.view(np.int16)).cuda().view(cuda.bfloat16)
    vt = cuda.from_numpy(vb.view(np.int16)).cuda().view(cuda.bfloat16)
    slots, slots_d = make_slots(cuda, n, nb, 4)
    layer.append(kt, vt, slots_d)
    pi = oracle_pi(layer)
    for which, bits in ((0, 3), (1, 4)):
        out = layer.dequantize(which, slots_d).cpu().numpy().astype(np.float64)
        c32, _ = ocb.codebook_fp32(D, bits)
        fields = page_fields(layer, which, (layer.k_cache if which == 0 else layer.v_cache).cpu().numpy())
        for h in range(H):
            codes, gamma = slot_fields(fields, slots, h)[:2]
            ref = oq.dequantize(codes, gamma, pi, c32)
            err = np.max(np.abs(out[:, h] - ref), axis=-1) / np.max(np.abs(ref), axis=-1)
            assert np.max(err) < 1e-5


@pytest.mark.parametrize("kind", ["dense_bulk", "hadamard_bulk", "small_mixed"])
def test_append_layers_equals_per_layer_appends(cuda, tqlib, kind):
    """tq_quantize_append_layers (the layers after the first launched as programmatic
    dependents of the previous layer's kernel, without waiting for it) writes exactly
    the pages of one tq_quantize_append per layer: the tensor-core and staged bulk
    kernels, and a small append over a mix of packed, QJL, dense and bf16 layers."""
    tq, torch = tqlib, cuda
    H = 8
    if kind == "small_mixed":
        n, nb = 37, 8
        fmts = [dict(seed=1, layer=0), dict(kv_format="bf16"), dict(bits_k=2, bits_v=4, qjl=True, seed=1, layer=2),
                dict(rot_kind=tq.TQ_ROT_DENSE, seed=1, layer=3), dict(bits_k=3, bits_v=3, seed=1, layer=4)]
    else:
        n, nb = 3100, 200  # 24,800 vectors per tensor: the bulk kernels
        rk = tq.TQ_ROT_DENSE if kind == "dense_bulk" else tq.TQ_ROT_HADAMARD
        fmts = [dict(rot_kind=rk, seed=7, layer=l, bits_k=b, bits_v=b) for l, b in enumerate((4, 3, 2, 4))]
    slots, slots_d = make_slots(cuda, n, nb, 5, skip_every=11)
    gen = torch.Generator(device="cuda").manual_seed(9)
    ks = [torch.randn(n, H, D, generator=gen, device="cuda").to(torch.bfloat16) for _ in fmts]
    vs = [torch.randn(n, H, D, generator=gen, device="cuda").to(torch.bfloat16) for _ in fmts]
    batched = [tq.Layer(nb, H, fill=0xA5, **f) for f in fmts]
    single = [tq.Layer(nb, H, fill=0xA5, **f) for f in fmts]
    tq.append_layers(batched, ks, vs, slots_d)
    for ly, k, v in zip(single, ks, vs):
        ly.append(k, v, slots_d)
    torch.cuda.synchronize()
    assert tq.get_device_status() == 0
    for a, b in zip(batched, single):
        assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.v_cache, b.v_cache)
    # a shared cache is rejected before anything is launched
    with pytest.raises(tq.TQError):
        tq.append_layers([batched[0], batched[0]], ks[:2], vs[:2], slots_d)


def _random_append_case(i):
    """Seeded random append configuration i: heads, tokens (some past the bulk kernels'
    24,576-vector threshold), key / value bits, rotation kind, QJL keys, input dtype,
    skipped slots, data."""
    r = np.random.default_rng(2000 + i)
    H = int(r.choice([1, 2, 4, 8]))
    n = int(r.integers(1, 900)) if r.random() < 0.6 else int(24576 // H + r.integers(1, 400))
    dense = bool(r.random() < 0.35)
    return dict(H=H, n=n, bits_k=int(r.choice([2, 3, 4])), bits_v=int(r.choice([2, 3, 4])), dense=dense,
                qjl=bool(r.random() < 0.2), f32=bool(r.random() < 0.25), skip=int(r.choice([0, 7, 37])),
                lognormal=bool(r.random() < 0.5), seed=40 + i)


@pytest.mark.parametrize("i", range(10))
def test_randomized_append_configurations(cuda, tqlib, i):
    """Ten seeded random appends against the oracle's quantizer: codes equal except
    within 1e-5 of a boundary, gamma within 2e-6 relative, skipped slots untouched."""
    tq = tqlib
    c = _random_append_case(i)
    print(c)
    H, n = c["H"], c["n"]
    nb = n // 16 + 3
    rot = tq.TQ_ROT_DENSE if c["dense"] else tq.TQ_ROT_HADAMARD
    layer = tq.Layer(nb, H, bits_k=c["bits_k"], bits_v=c["bits_v"], qjl=c["qjl"], rot_kind=rot, seed=c["seed"],
                     layer=3, qjl_seed=c["seed"] + 1, fill=0x5A)
    if c["lognormal"]:
        kb, vb = workloads.lognormal_channel_kv(c["seed"], n, H, D)
    else:
        kb, vb = workloads.scaled_gaussian_kv(c["seed"], n, H, D)
    if c["f32"]:
        kx, vx = workloads.bf16_to_f32(kb), workloads.bf16_to_f32(vb)
        kt, vt = cuda.from_numpy(kx).cuda(), cuda.from_numpy(vx).cuda()
        kx, vx = kx.astype(np.float64), vx.astype(np.float64)
    else:
        kt, vt = _bf16_dev(cuda, kb), _bf16_dev(cuda, vb)
        kx, vx = oq.bf16_bits_to_f64(kb), oq.bf16_bits_to_f64(vb)
    slots, slots_d = make_slots(cuda, n, nb, c["seed"] + 2, skip_every=c["skip"])
    layer.append(kt, vt, slots_d)
    assert tq.get_device_status() == 0
    pi = (orot.dense_rotation_seeded if c["dense"] else orot.hadamard_rotation_seeded)(c["seed"], 3, D)
    keep = slots >= 0
    written = np.zeros(nb * 16, bool)
    written[slots[keep]] = True
    for which, x, pool, bits in ((0, kx, layer.k_cache, c["bits_k"]), (1, vx, layer.v_cache, c["bits_v"])):
        c32, b32 = ocb.codebook_fp32(D, bits)
        host = pool.cpu().numpy()
        fields = page_fields(layer, which, host)
        for h in range(H):
            idx, gamma, y = oq.quantize(x[keep, h], pi, c32, b32)
            codes, g_gpu = slot_fields(fields, slots[keep], h)[:2]  # (QJL pages add signs and rho)
            ok, _ = tie_band_ok(y, codes, idx, b32, 1e-5)
            assert ok, "code mismatch outside the tie band"
            same = np.all(codes == idx, axis=-1)
            assert np.all(np.abs(g_gpu[same] - gamma[same]) <= 2e-6 * np.abs(gamma[same]) + 1e-30)
        if not (which == 0 and c["qjl"]):
            rec = opack_record_view(host, nb, H, bits)
            assert np.all(rec[~written.reshape(nb, 16)] == 0x5A)
