"""GPU parity of decode attention on the packed (and bf16) cache against the
oracle's exact softmax attention over the GPU's own cache."""
import math

import numpy as np
import pytest

import workloads
from oracle import attention as oa, quantize as oq
from tests._gpu_util import D, max_rel_err, oracle_layer

pytestmark = pytest.mark.gpu

TOL_F32 = 2e-3
TOL_BF16 = 5e-3


def to_dev(cuda, arr, bf16=False):
    if bf16:
        return cuda.from_numpy(np.ascontiguousarray(arr).view(np.int16)).cuda().view(cuda.bfloat16)
    return cuda.from_numpy(np.ascontiguousarray(arr)).cuda()


def fill_cache(cuda, layer, kx, vx, block_table, ctx, bf16):
    """Append token t of sequence b at its block-table slot (one batched call)."""
    bsz = block_table.shape[0]
    slots = []
    ks, vs = [], []
    for b in range(bsz):
        pos = np.arange(ctx[b])
        slots.append(workloads.slot_mapping(block_table[b:b + 1], pos[None, :])[0])
        ks.append(kx[b, : ctx[b]])
        vs.append(vx[b, : ctx[b]])
    slots = np.concatenate(slots).astype(np.int64)
    k = np.concatenate(ks)
    v = np.concatenate(vs)
    layer.append(to_dev(cuda, k, bf16), to_dev(cuda, v, bf16), cuda.from_numpy(slots).cuda())


def run_case(cuda, tq, *, B, Hq, Hkv, ctx, bits_k=4, bits_v=4, qjl=False, rot=1, bf16=True, kv_format="packed",
             data="gauss", seed=0, num_splits=0, q_f32=False, out_f32=True, extra_blocks=3):
    ctx = np.asarray(ctx, np.int32)
    mb = int(max(1, math.ceil(ctx.max() / 16)))
    bt, nb = workloads.shuffled_block_table(seed + 1, B, mb, num_blocks=B * mb + extra_blocks)
    tmax = mb * 16
    if data == "lognormal":
        kb, vb = workloads.lognormal_channel_kv(seed, B * tmax, Hkv, D)
    elif data == "heavy":
        kb, vb = workloads.heavy_tail_kv(seed, B * tmax, Hkv, D)
    else:
        kb, vb = workloads.scaled_gaussian_kv(seed, B * tmax, Hkv, D)
    kb = kb.reshape(B, tmax, Hkv, D)
    vb = vb.reshape(B, tmax, Hkv, D)
    layer = tq.Layer(nb, Hkv, kv_format=kv_format, bits_k=bits_k, bits_v=bits_v, qjl=qjl, rot_kind=rot,
                     seed=seed + 7, layer=seed % 5, qjl_seed=seed + 11)
    if bf16:
        fill_cache(cuda, layer, kb, vb, bt, ctx, True)
    else:
        fill_cache(cuda, layer, workloads.bf16_to_f32(kb), workloads.bf16_to_f32(vb), bt, ctx, False)
    qf = workloads.queries(seed + 3, B, Hq, D, dtype="f32" if q_f32 else "bf16")
    qd = to_dev(cuda, qf, bf16=not q_f32)
    sm = 1.0 / math.sqrt(D)
    out = layer.decode(qd, cuda.from_numpy(bt).cuda(), cuda.from_numpy(ctx).cuda(), sm_scale=sm,
                       out_dtype=cuda.float32 if out_f32 else cuda.bfloat16, num_splits=num_splits)
    cuda.cuda.synchronize()
    assert tq.get_device_status() == 0
    qx = qf.astype(np.float64) if q_f32 else oq.bf16_bits_to_f64(qf)
    kp, vp = layer.k_cache.cpu().numpy(), layer.v_cache.cpu().numpy()
    if kv_format == "packed":
        ref = oa.decode_packed(qx, kp, vp, oracle_layer(layer), nb, Hkv, bt, ctx, sm)
    else:
        ref = oa.decode_bf16(qx, kp.view(np.uint16), vp.view(np.uint16), nb, Hkv, bt, ctx, sm)
    return out.float().cpu().numpy(), ref, layer


def assert_close(out, ref, tol, ctx):
    live = np.asarray(ctx) > 0
    err = max_rel_err(out[live], ref[live])
    print("max rel err %.3e (tol %.1e)" % (err, tol))
    assert err <= tol
    assert np.all(out[~live] == 0.0)


def test_tiny_single_head_fp32(cuda, tqlib):
    # 1 seq, 1 KV head, 256 tokens, fp32 K/V with 4 outlier channels x20, 4-bit, Hadamard seed 0
    tq = tqlib
    k, v, q, _ = workloads.tiny_kv(seed=0)
    layer = tq.Layer(16, 1, seed=0, layer=0)
    slots = np.arange(256, dtype=np.int64)
    layer.append(to_dev(cuda, k), to_dev(cuda, v), cuda.from_numpy(slots).cuda())
    bt = np.arange(16, dtype=np.int32)[None, :]
    ctx = np.array([256], np.int32)
    out = layer.decode(to_dev(cuda, q), cuda.from_numpy(bt).cuda(), cuda.from_numpy(ctx).cuda())
    cuda.cuda.synchronize()
    ref = oa.decode_packed(q.astype(np.float64), layer.k_cache.cpu().numpy(), layer.v_cache.cpu().numpy(),
                           oracle_layer(layer), 16, 1, bt, ctx, 1 / math.sqrt(D))
    assert_close(out.cpu().numpy(), ref, TOL_F32, ctx)


@pytest.mark.parametrize("splits", [0, 3])
def test_gqa_lognormal_bf16(cuda, tqlib, splits):
    out, ref, _ = run_case(cuda, tqlib, B=3, Hq=8, Hkv=2, ctx=[1, 100, 333], data="lognormal", num_splits=splits)
    assert_close(out, ref, TOL_BF16, [1, 100, 333])


def test_group8_heavy_tail_k3v4(cuda, tqlib):
    out, ref, _ = run_case(cuda, tqlib, B=2, Hq=16, Hkv=2, ctx=[500, 77], bits_k=3, bits_v=4, data="heavy", seed=2)
    assert_close(out, ref, TOL_BF16, [500, 77])


@pytest.mark.parametrize("bk,bv", [(2, 2), (2, 3), (3, 3), (4, 2)])
def test_other_bit_widths(cuda, tqlib, bk, bv):
    out, ref, _ = run_case(cuda, tqlib, B=2, Hq=4, Hkv=2, ctx=[45, 160], bits_k=bk, bits_v=bv, seed=3)
    assert_close(out, ref, TOL_BF16, [45, 160])


def test_qjl_keys(cuda, tqlib):
    out, ref, _ = run_case(cuda, tqlib, B=2, Hq=8, Hkv=2, ctx=[300, 129], bits_k=2, bits_v=4, qjl=True, seed=4)
    assert_close(out, ref, TOL_BF16, [300, 129])


def test_lmdeploy_layout_k3_qjl_v2(cuda, tqlib):
    """LMDeploy's layout ([P1] §LMDeploy): 3-bit keys with the QJL residual, 2-bit values."""
    out, ref, _ = run_case(cuda, tqlib, B=2, Hq=8, Hkv=2, ctx=[257, 90], bits_k=3, bits_v=2, qjl=True, seed=12)
    assert_close(out, ref, TOL_BF16, [257, 90])


def test_dense_rotation_layer(cuda, tqlib):
    out, ref, _ = run_case(cuda, tqlib, B=1, Hq=8, Hkv=2, ctx=[300], rot=tqlib.TQ_ROT_DENSE, seed=5, q_f32=True)
    assert_close(out, ref, TOL_BF16, [300])


def test_bf16_layer(cuda, tqlib):
    out, ref, _ = run_case(cuda, tqlib, B=2, Hq=8, Hkv=2, ctx=[70, 257], kv_format="bf16", seed=6)
    assert_close(out, ref, TOL_BF16, [70, 257])


def test_fp32_inputs_fp32_tolerance(cuda, tqlib):
    out, ref, _ = run_case(cuda, tqlib, B=2, Hq=4, Hkv=1, ctx=[200, 31], bf16=False, q_f32=True, seed=7)
    assert_close(out, ref, TOL_F32, [200, 31])


def test_sixteen_heads_per_kv_head(cuda, tqlib):
    out, ref, _ = run_case(cuda, tqlib, B=1, Hq=16, Hkv=1, ctx=[190], seed=8)
    assert_close(out, ref, TOL_BF16, [190])


def test_empty_and_single_token_contexts(cuda, tqlib):
    out, ref, _ = run_case(cuda, tqlib, B=3, Hq=4, Hkv=2, ctx=[0, 1, 17], seed=9)
    assert_close(out, ref, TOL_BF16, [0, 1, 17])


def test_split_count_invariance(cuda, tqlib):
    outs = []
    for s in (1, 2, 5, 16, 64):
        out, ref, _ = run_case(cuda, tqlib, B=2, Hq=8, Hkv=2, ctx=[1000, 411], seed=10, num_splits=s)
        outs.append(out)
    for o in outs[1:]:
        assert max_rel_err(o, outs[0]) < 2e-5


def test_many_splits_use_the_combine_kernel(cuda, tqlib):
    """More than 128 splits of a unit are merged by the separate combine kernel
    instead of the decode kernel's own merge: same result as a fused call within the
    split-invariance bound, and the oracle's within tolerance (one sequence of 3,300
    tokens, 207 blocks, 200 splits, and a shorter one whose later splits are empty)."""
    ctx = [3300, 170]
    out200, ref, _ = run_case(cuda, tqlib, B=2, Hq=8, Hkv=2, ctx=ctx, seed=12, num_splits=200)
    assert_close(out200, ref, TOL_BF16, ctx)
    out16, _, _ = run_case(cuda, tqlib, B=2, Hq=8, Hkv=2, ctx=ctx, seed=12, num_splits=16)
    assert max_rel_err(out200, out16) < 2e-5


def test_bad_block_table_entry_is_flagged(cuda, tqlib):
    tq = tqlib
    layer = tq.Layer(4, 1)
    q = cuda.zeros((1, 1, D), dtype=cuda.float32).cuda()
    bt = cuda.tensor([[0, 99]], dtype=cuda.int32).cuda()
    ctx = cuda.tensor([20], dtype=cuda.int32).cuda()
    layer.decode(q, bt, ctx)
    assert tq.get_device_status() & tq.TQ_DEV_BAD_BLOCK
    ctx = cuda.tensor([1000], dtype=cuda.int32).cuda()
    layer.decode(q, bt[:, :1].contiguous(), ctx)
    assert tq.get_device_status() & tq.TQ_DEV_BAD_CONTEXT


def spread_pairs(B, Hkv, n=8):
    """n (sequence, KV head) pairs spread over the first, middle and last units."""
    units = np.unique(np.linspace(0, B * Hkv - 1, n).round().astype(int))
    return tuple((int(u) // Hkv, int(u) % Hkv) for u in units)


def test_llama8b_shape_full_size_sampled(cuda, tqlib):
    """Batch 16, 32/8 heads, context 8192, lognormal channels, shuffled table;
    the oracle checks 8 sampled (sequence, KV head) pairs of the full-size run, with
    fp32 outputs and with the bf16 outputs the benchmark produces."""
    tq = tqlib
    B, Hq, Hkv, T = 16, 32, 8, 8192
    mb = T // 16
    bt, nb = workloads.shuffled_block_table(21, B, mb + 1)
    layer = tq.Layer(nb, Hkv, seed=0, layer=0)
    torch = cuda
    gen = torch.Generator(device="cuda").manual_seed(5)
    scale_k = torch.exp(torch.randn(Hkv, D, generator=gen, device="cuda"))
    scale_v = torch.exp(torch.randn(Hkv, D, generator=gen, device="cuda"))
    k = (torch.randn(B * T, Hkv, D, generator=gen, device="cuda") * scale_k).to(torch.bfloat16)
    v = (torch.randn(B * T, Hkv, D, generator=gen, device="cuda") * scale_v).to(torch.bfloat16)
    slots = workloads.prefill_slots(bt, T)
    layer.append(k, v, torch.from_numpy(slots).cuda())
    ctx = np.full(B, T, np.int32)
    q = torch.randn(B, Hq, D, generator=gen, device="cuda").to(torch.bfloat16)
    out = layer.decode(q, torch.from_numpy(bt).cuda(), torch.from_numpy(ctx).cuda(), out_dtype=torch.float32)
    out16 = layer.decode(q, torch.from_numpy(bt).cuda(), torch.from_numpy(ctx).cuda(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert tq.get_device_status() == 0
    kp, vp = layer.k_cache.cpu().numpy(), layer.v_cache.cpu().numpy()
    ol = oracle_layer(layer)
    qx = q.float().cpu().numpy().astype(np.float64)
    o = out.cpu().numpy()
    o16 = out16.float().cpu().numpy()
    errs, errs16 = [], []
    for b, kvh in spread_pairs(B, Hkv):
        f = oa.gather_packed(kp, vp, ol, nb, Hkv, D, bt[b], T, kvh)
        for h in range(kvh * 4, kvh * 4 + 4):
            s = (1 / math.sqrt(D)) * (f["k_hat"] @ qx[b, h])
            ref = oa.softmax_weights(s) @ f["v_hat"]
            errs.append(max_rel_err(o[b, h][None], ref[None]))
            errs16.append(max_rel_err(o16[b, h][None], ref[None]))
    print("sampled max rel err %.3e (fp32 out), %.3e (bf16 out)" % (max(errs), max(errs16)))
    assert max(errs) <= TOL_BF16
    # the bf16 store is the fp32 result rounded to nearest even, element for element ...
    assert torch.equal(out16, out.to(torch.bfloat16))
    # ... which adds at most half a bf16 ulp (2^-8 of the element) to the error
    assert max(errs16) <= TOL_BF16 + 2.0 ** -8


def test_late_max_jump_after_large_weight(cuda, tqlib):
    """Rescale path of the online softmax: token A (large value norm) sits just
    under the lazy-rescale threshold and sets the value reference, then token B
    moves the running maximum by more than the threshold while its own weight
    stays below the rescaled reference.  One chunk per unit, fp32 throughout."""
    tq = tqlib
    rng = np.random.default_rng(17)
    Hkv, Hq, T = 1, 4, 128
    q = rng.standard_normal((1, Hq, D))
    sm = 1.0 / math.sqrt(D)
    qn = q[0, 0] / np.linalg.norm(q[0, 0])
    per_unit = np.linalg.norm(q[0, 0]) * sm / math.log(2.0)  # base-2 logit per unit of k along q
    k = rng.standard_normal((1, T, Hkv, D)) * 0.02
    v = rng.standard_normal((1, T, Hkv, D))
    k[0, 3, 0] = qn * (0.5 / per_unit)    # block 0: running max 1
    k[0, 40, 0] = qn * (20.5 / per_unit)  # under max + 20: weight ~2^19.5
    v[0, 40, 0] *= 10.0
    k[0, 90, 0] = qn * (21.6 / per_unit)  # over max + 20: the maximum moves to 22
    bt, nb = workloads.shuffled_block_table(3, 1, T // 16, num_blocks=T // 16 + 2)
    layer = tq.Layer(nb, Hkv, seed=4, layer=1)
    fill_cache(cuda, layer, k.astype(np.float32), v.astype(np.float32), bt, [T], False)
    ctx = np.array([T], np.int32)
    out = layer.decode(to_dev(cuda, q.astype(np.float32)), cuda.from_numpy(bt).cuda(), cuda.from_numpy(ctx).cuda(),
                       sm_scale=sm, out_dtype=cuda.float32, num_splits=1)
    cuda.cuda.synchronize()
    assert tq.get_device_status() == 0
    kp, vp = layer.k_cache.cpu().numpy(), layer.v_cache.cpu().numpy()
    ol = oracle_layer(layer)
    f = oa.gather_packed(kp, vp, ol, nb, Hkv, D, bt[0], T, 0)
    u = (f["k_hat"] @ q[0, 0]) * sm / math.log(2.0)
    # the scenario holds on the quantized cache
    assert math.ceil(u[:16].max()) == 1 and u[40] < 21.0 < u[90] and math.ceil(u[90]) == 22
    assert f["v_gamma"][40] > 4.0 * f["v_gamma"][90]
    ref = oa.decode_packed(q, kp, vp, ol, nb, Hkv, bt, ctx, sm)
    assert_close(out.cpu().numpy(), ref, TOL_F32, ctx)


def test_workspace_reused_across_shapes(cuda, tqlib):
    """One zero-filled workspace serves calls of different shapes and layers in
    turn: the per-unit chunk counters return to zero after every call."""
    tq = tqlib
    sm = 1.0 / math.sqrt(D)
    ws = cuda.zeros(8 << 20, dtype=cuda.uint8, device="cuda")
    cases = [dict(B=2, Hq=8, Hkv=2, ctx=[300, 77], seed=31), dict(B=3, Hq=32, Hkv=4, ctx=[900, 5, 400], seed=32),
             dict(B=2, Hq=8, Hkv=2, ctx=[300, 77], seed=31)]
    for cs in cases:
        out_ref, ref, layer = run_case(cuda, tq, B=cs["B"], Hq=cs["Hq"], Hkv=cs["Hkv"], ctx=cs["ctx"], seed=cs["seed"])
        ctx = np.asarray(cs["ctx"], np.int32)
        mb = int(math.ceil(ctx.max() / 16))
        bt, _ = workloads.shuffled_block_table(cs["seed"] + 1, cs["B"], mb, num_blocks=cs["B"] * mb + 3)
        q = to_dev(cuda, workloads.queries(cs["seed"] + 3, cs["B"], cs["Hq"], D, dtype="bf16"), bf16=True)
        need = layer.workspace_bytes(cs["B"], cs["Hq"], mb)
        assert need <= ws.numel()
        for _ in range(2):
            out = layer.decode(q, cuda.from_numpy(bt).cuda(), cuda.from_numpy(ctx).cuda(), sm_scale=sm,
                               out_dtype=cuda.float32, workspace=ws)
            cuda.cuda.synchronize()
            assert tq.get_device_status() == 0
            assert_close(out.cpu().numpy(), ref, TOL_BF16, ctx)
        # the counter region is zero again after the calls
        assert int(ws[:65536].count_nonzero().item()) == 0


@pytest.mark.parametrize("kind", ["hadamard", "dense", "qjl"])
def test_append_decode_equals_separate_calls(cuda, tqlib, kind):
    """tq_append_decode (the decode launched as a programmatic dependent of the append,
    its prologue overlapping the append) gives bit-identical outputs and caches to
    tq_quantize_append followed by tq_decode_attention, step after step."""
    tq = tqlib
    B, Hq, Hkv, T = 4, 16, 4, 320
    mb = T // 16
    bt, nb = workloads.shuffled_block_table(5, B, mb, num_blocks=B * mb + 2)
    kb, vb = workloads.scaled_gaussian_kv(9, B * T, Hkv, D)
    kb, vb = kb.reshape(B, T, Hkv, D), vb.reshape(B, T, Hkv, D)
    kw = dict(bits_k=2 if kind == "qjl" else 4, bits_v=4, qjl=kind == "qjl",
              rot_kind=tq.TQ_ROT_DENSE if kind == "dense" else tq.TQ_ROT_HADAMARD, seed=3, layer=1, qjl_seed=4)
    la, lb = tq.Layer(nb, Hkv, **kw), tq.Layer(nb, Hkv, **kw)
    ctx0 = np.array([200, 7, 150, 33], np.int32)
    for layer in (la, lb):
        fill_cache(cuda, layer, kb, vb, bt, ctx0, True)
    bt_d = cuda.from_numpy(bt).cuda()
    for step in range(3):
        pos = ctx0 + step
        slots = workloads.slot_mapping(bt, pos[:, None])[:, 0].astype(np.int64)
        knew = to_dev(cuda, kb[np.arange(B), pos], True)
        vnew = to_dev(cuda, vb[np.arange(B), pos], True)
        slots_d = cuda.from_numpy(slots).cuda()
        q = to_dev(cuda, workloads.queries(20 + step, B, Hq, D), True)
        ctx_d = cuda.from_numpy(pos + 1).cuda()
        out_a = la.append_decode(knew, vnew, slots_d, q, bt_d, ctx_d, out_dtype=cuda.float32)
        lb.append(knew, vnew, slots_d)
        out_b = lb.decode(q, bt_d, ctx_d, out_dtype=cuda.float32)
        cuda.cuda.synchronize()
        assert tq.get_device_status() == 0
        assert np.array_equal(out_a.cpu().numpy(), out_b.cpu().numpy())
        assert np.array_equal(la.k_cache.cpu().numpy(), lb.k_cache.cpu().numpy())
        assert np.array_equal(la.v_cache.cpu().numpy(), lb.v_cache.cpu().numpy())


def _sampled_err(tq, layer, out, q, bt, ctx, pairs, sm, g):
    """Max relative error of out over the heads of sampled (sequence, KV head) pairs
    against exact attention over the GPU's own cache (oracle gathers per pair)."""
    kp, vp = layer.k_cache.cpu().numpy(), layer.v_cache.cpu().numpy()
    nb, hkv = layer.num_blocks, layer.num_kv_heads
    qx = q.float().cpu().numpy().astype(np.float64)
    o = out.float().cpu().numpy()
    errs = []
    if not layer.packed:
        for b, kvh in pairs:
            k, v = oa.gather_bf16(kp.view(np.uint16), vp.view(np.uint16), nb, hkv, D, bt[b], int(ctx[b]), kvh)
            for h in range(kvh * g, (kvh + 1) * g):
                errs.append(max_rel_err(o[b, h][None], oa.softmax_attention(qx[b, h], k, v, sm)[None]))
        return max(errs)
    ol = oracle_layer(layer)
    for b, kvh in pairs:
        f = oa.gather_packed(kp, vp, ol, nb, hkv, D, bt[b], int(ctx[b]), kvh)
        for h in range(kvh * g, (kvh + 1) * g):
            if ol.qjl:
                from oracle import qjl as oqjl
                s = sm * oqjl.estimate(qx[b, h], ol.pi, ol.cb_k, f["k_idx"], f["k_gamma"], f["k_signs"], f["k_rho"],
                                       ol.qjl_s)
            else:
                s = sm * (f["k_hat"] @ qx[b, h])
            errs.append(max_rel_err(o[b, h][None], (oa.softmax_weights(s) @ f["v_hat"])[None]))
    return max(errs)


def _gpu_kv(torch, gen, n, hkv, heavy):
    """bf16 [n, hkv, d] N(0, 1) K and V; heavy: each element replaced with probability
    0.01 by an unscaled Student-t(3) draw (z / sqrt(chi2_3 / 3))."""
    out = []
    for _ in range(2):
        x = torch.randn(n, hkv, D, generator=gen, device="cuda")
        if heavy:
            mask = torch.rand(n, hkv, D, generator=gen, device="cuda") < 0.01
            chi = sum(torch.randn(n, hkv, D, generator=gen, device="cuda") ** 2 for _ in range(3))
            t3 = torch.randn(n, hkv, D, generator=gen, device="cuda") / torch.sqrt(chi / 3.0)
            x = torch.where(mask, t3, x)
            del mask, chi, t3
        out.append(x.to(torch.bfloat16))
        del x
    return out


def test_config3_shape_full_size_sampled(cuda, tqlib):
    """Batch 4, 64 query / 8 KV heads (groups of 8), context 131,072 (8192 blocks per
    sequence), 3-bit keys / 4-bit values, N(0, 1) with 1 % Student-t(3) elements,
    shuffled table; sampled (sequence, KV head) pairs of the full-size run."""
    tq, torch = tqlib, cuda
    B, Hq, Hkv, T = 4, 64, 8, 131072
    bt, nb = workloads.shuffled_block_table(31, B, T // 16)
    layer = tq.Layer(nb, Hkv, bits_k=3, bits_v=4, seed=3, layer=2)
    gen = torch.Generator(device="cuda").manual_seed(33)
    k, v = _gpu_kv(torch, gen, B * T, Hkv, heavy=True)
    layer.append(k, v, torch.from_numpy(workloads.prefill_slots(bt, T)).cuda())
    del k, v
    ctx = np.full(B, T, np.int32)
    q = torch.randn(B, Hq, D, generator=gen, device="cuda").to(torch.bfloat16)
    out = layer.decode(q, torch.from_numpy(bt).cuda(), torch.from_numpy(ctx).cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tq.get_device_status() == 0
    err = _sampled_err(tq, layer, out, q, bt, ctx, spread_pairs(B, Hkv), 1 / math.sqrt(D), Hq // Hkv)
    print("config 3 sampled max rel err %.3e" % err)
    assert err <= TOL_BF16


@pytest.mark.parametrize("variant", ["packed", "qjl", "bf16"])
def test_config5_layers_full_size_sampled(cuda, tqlib, variant):
    """Batch 8, 32 query / 8 KV heads, context 100,000 (6250 blocks per sequence) for
    the three layer kinds of the mixed-precision model: a 4/4 packed layer, the
    variant with 2-bit + QJL keys and 4-bit values, and a bf16 boundary layer."""
    tq, torch = tqlib, cuda
    B, Hq, Hkv, T = 8, 32, 8, 100000
    bt, nb = workloads.shuffled_block_table(51, B, -(-T // 16))
    if variant == "bf16":
        layer = tq.Layer(nb, Hkv, kv_format="bf16")
    elif variant == "qjl":
        layer = tq.Layer(nb, Hkv, bits_k=2, bits_v=4, qjl=True, seed=5, layer=11, qjl_seed=9)
    else:
        layer = tq.Layer(nb, Hkv, seed=5, layer=11)
    gen = torch.Generator(device="cuda").manual_seed(55)
    k, v = _gpu_kv(torch, gen, B * T, Hkv, heavy=False)
    layer.append(k, v, torch.from_numpy(workloads.prefill_slots(bt, T)).cuda())
    del k, v
    ctx = np.full(B, T, np.int32)
    q = torch.randn(B, Hq, D, generator=gen, device="cuda").to(torch.bfloat16)
    out = layer.decode(q, torch.from_numpy(bt).cuda(), torch.from_numpy(ctx).cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tq.get_device_status() == 0
    err = _sampled_err(tq, layer, out, q, bt, ctx, spread_pairs(B, Hkv), 1 / math.sqrt(D), Hq // Hkv)
    print("config 5 %s sampled max rel err %.3e" % (variant, err))
    assert err <= TOL_BF16


def test_config4_dense_layer_full_size(cuda, tqlib):
    """One layer of the dense-rotation workload at full size: 11,000 prefilled bf16
    tokens x 8 KV heads scaled by lambda = 2.7 through the tensor-core append (a ragged
    last block), then batch-1 decode with 32 query heads; every KV head checked."""
    tq, torch = tqlib, cuda
    B, Hq, Hkv, T = 1, 32, 8, 11000
    bt, nb = workloads.shuffled_block_table(41, B, -(-T // 16))
    layer = tq.Layer(nb, Hkv, rot_kind=tq.TQ_ROT_DENSE, seed=36, layer=4)
    gen = torch.Generator(device="cuda").manual_seed(44)
    k, v = _gpu_kv(torch, gen, B * T, Hkv, heavy=False)
    k, v = (k.float() * 2.7).to(torch.bfloat16), (v.float() * 2.7).to(torch.bfloat16)
    layer.append(k, v, torch.from_numpy(workloads.prefill_slots(bt, T)).cuda())
    ctx = np.full(B, T, np.int32)
    q = torch.randn(B, Hq, D, generator=gen, device="cuda").to(torch.bfloat16)
    out = layer.decode(q, torch.from_numpy(bt).cuda(), torch.from_numpy(ctx).cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tq.get_device_status() == 0
    err = _sampled_err(tq, layer, out, q, bt, ctx, tuple((0, h) for h in range(Hkv)), 1 / math.sqrt(D), Hq // Hkv)
    print("config 4 layer max rel err %.3e" % err)
    assert err <= TOL_BF16


def test_incremental_dequant_baseline_attends_the_same_tokens(cuda, tqlib):
    """The incremental-dequant baseline (a bf16 running cache filled from
    tq_dequantize, then bf16 decode) attends the same tokens as the fused decode on
    the packed cache: equal up to the bf16 rounding of the dequantized values."""
    tq, torch = tqlib, cuda
    B, Hq, Hkv, T = 4, 16, 4, 700
    bt, nb = workloads.shuffled_block_table(81, B, -(-T // 16))
    layer = tq.Layer(nb, Hkv, seed=2, layer=6)
    shadow = tq.Layer(nb, Hkv, kv_format="bf16")
    kb, vb = workloads.scaled_gaussian_kv(82, B * T, Hkv, D)  # N(0, 1): logits of order 1
    slots = torch.from_numpy(workloads.prefill_slots(bt, T)).cuda()
    layer.append(torch.from_numpy(kb.view(np.int16)).cuda().view(torch.bfloat16),
                 torch.from_numpy(vb.view(np.int16)).cuda().view(torch.bfloat16), slots)
    shadow.append(layer.dequantize(0, slots, out_dtype=torch.bfloat16),
                  layer.dequantize(1, slots, out_dtype=torch.bfloat16), slots)
    q = torch.from_numpy(workloads.queries(83, B, Hq, D).view(np.int16)).cuda().view(torch.bfloat16)
    ctx = torch.from_numpy(np.full(B, T, np.int32)).cuda()
    bt_d = torch.from_numpy(bt).cuda()
    o_packed = layer.decode(q, bt_d, ctx, out_dtype=torch.float32).cpu().numpy()
    o_shadow = shadow.decode(q, bt_d, ctx, out_dtype=torch.float32).cpu().numpy()
    assert tq.get_device_status() == 0
    err = max_rel_err(o_shadow.reshape(-1, D), o_packed.reshape(-1, D))
    print("incremental-dequant baseline vs fused: max rel err %.3e" % err)
    assert err <= 1e-2  # bf16 rounding of the dequantized K/V; a wrong token would be O(1)


def test_padded_block_table_splits_the_context(cuda, tqlib):
    """A block-table row far wider than the context (a table padded to a maximum
    length, the padding set to -1 so that reading it would be flagged) is split over
    the context: with the same split count the output equals, bit for bit, the one
    for a table cut to the longest context, and matches the oracle."""
    tq = tqlib
    B, Hq, Hkv, S = 3, 8, 2, 6
    ctx = np.array([517, 300, 64], np.int32)
    out_t, ref, layer = run_case(cuda, tq, B=B, Hq=Hq, Hkv=Hkv, ctx=ctx, seed=9, num_splits=S)
    assert_close(out_t, ref, TOL_BF16, ctx)
    mb = int(math.ceil(ctx.max() / 16))
    bt, _ = workloads.shuffled_block_table(10, B, mb, num_blocks=B * mb + 3)  # the table run_case used
    padded = np.full((B, 8 * mb), -1, np.int32)
    padded[:, :mb] = bt
    qf = workloads.queries(9 + 3, B, Hq, D, dtype="bf16")
    out_p = layer.decode(to_dev(cuda, qf, bf16=True), cuda.from_numpy(padded).cuda(), cuda.from_numpy(ctx).cuda(),
                         sm_scale=1.0 / math.sqrt(D), out_dtype=cuda.float32, num_splits=S)
    cuda.cuda.synchronize()
    assert tq.get_device_status() == 0
    assert np.array_equal(out_p.cpu().numpy(), out_t)


def _random_case(i):
    """Seeded random decode configuration i: batch, KV heads, query heads per KV head
    (partial groups of 4 and 8 included), key / value bits, QJL keys, rotation kind,
    ragged contexts (empty ones included), split count, data and query precision."""
    r = np.random.default_rng(1000 + i)
    hkv = int(r.choice([1, 2, 4]))
    g = int(r.choice([1, 2, 3, 4, 5, 8, 12, 16]))
    B = int(r.integers(1, 4))
    ctx = [int(c) for c in r.integers(1, 700, size=B)]
    if B > 1 and r.random() < 0.3:  # an empty sequence beside live ones
        ctx[int(r.integers(0, B))] = 0
    qjl = bool(r.random() < 0.25)
    return dict(B=B, Hq=g * hkv, Hkv=hkv, ctx=ctx, bits_k=int(r.choice([2, 3, 4])), bits_v=int(r.choice([2, 3, 4])),
                qjl=qjl, rot=1 if r.random() < 0.75 else 2, data=str(r.choice(["gauss", "lognormal", "heavy"])),
                seed=20 + i, num_splits=int(r.choice([0, 0, 1, int(r.integers(2, 41))])),
                q_f32=bool(r.random() < 0.3))


@pytest.mark.parametrize("i", range(16))
def test_randomized_decode_configurations(cuda, tqlib, i):
    """Sixteen seeded random configurations against the oracle's exact attention over
    the GPU's own cache (bf16 inputs: the 5e-3 tolerance)."""
    kw = _random_case(i)
    if kw["rot"] == 2:
        kw["rot"] = tqlib.TQ_ROT_DENSE
    else:
        kw["rot"] = tqlib.TQ_ROT_HADAMARD
    print(kw)
    out, ref, _ = run_case(cuda, tqlib, **kw)
    assert_close(out, ref, TOL_BF16, kw["ctx"])


@pytest.mark.parametrize("bk,bv,f32,g", [(4, 4, False, 4), (3, 4, False, 4), (2, 2, True, 4), (4, 4, False, 8),
                                          (3, 4, False, 12)])
def test_decode_step_appends_and_attends(cuda, tqlib, bk, bv, f32, g):
    """tq_decode_step (the new token quantized by the decode kernel itself) against an
    append at the same slots followed by a decode, step after step: the new records
    follow the oracle's quantizer (codes except within 1e-5 of a boundary, gamma within
    2e-6), every other byte of the cache is the same, and the output matches the
    oracle's attention over the resulting cache."""
    from oracle import codebook as ocb
    from tests._gpu_util import oracle_pi, page_fields, slot_fields, tie_band_ok
    tq = tqlib
    B, Hkv, T = 4, 4, 320
    Hq = g * Hkv  # groups of 4, of 8 (two n-tiles), and of 12 (two head groups writing the same record)
    mb = T // 16 + 1
    bt, nb = workloads.shuffled_block_table(15, B, mb, num_blocks=B * mb + 2)
    # groups of 12 run on Gaussian data: with lognormal channels and 3-bit keys one output
    # row measures 5.3e-3 for the plain decode as well (the fp16 centroid tables)
    kb, vb = (workloads.lognormal_channel_kv if g != 12 else workloads.scaled_gaussian_kv)(16, B * T, Hkv, D)
    kb, vb = kb.reshape(B, T, Hkv, D), vb.reshape(B, T, Hkv, D)
    kw = dict(bits_k=bk, bits_v=bv, seed=5, layer=2)
    la, lb = tq.Layer(nb, Hkv, **kw), tq.Layer(nb, Hkv, **kw)
    ctx0 = np.array([200, 7, 0, 33], np.int32)  # sequence 2 starts empty
    for layer in (la, lb):
        fill_cache(cuda, layer, kb, vb, bt, ctx0, True)
    bt_d = cuda.from_numpy(bt).cuda()
    pi = oracle_pi(la)
    appended = []  # every slot written so far (its gamma may differ in the last bits between the paths)
    for step in range(3):
        pos = ctx0 + step
        slots = workloads.slot_mapping(bt, pos[:, None])[:, 0].astype(np.int64)
        appended.extend(int(x) for x in slots)
        kx, vx = kb[np.arange(B), pos], vb[np.arange(B), pos]  # [B][Hkv][D] bf16 bits
        if f32:
            knew = cuda.from_numpy(workloads.bf16_to_f32(kx)).cuda()
            vnew = cuda.from_numpy(workloads.bf16_to_f32(vx)).cuda()
        else:
            knew, vnew = to_dev(cuda, kx, True), to_dev(cuda, vx, True)
        q = to_dev(cuda, workloads.queries(40 + step, B, Hq, D), True)
        ctx_d = cuda.from_numpy(pos + 1).cuda()
        out_a = la.decode_step(knew, vnew, q, bt_d, ctx_d, out_dtype=cuda.float32)
        lb.append(knew, vnew, cuda.from_numpy(slots).cuda())
        lb.decode(q, bt_d, ctx_d, out_dtype=cuda.float32)
        cuda.cuda.synchronize()
        assert tq.get_device_status() == 0
        # the new records against the oracle's quantizer, the rest of the cache unchanged
        for which, x, bits, pa, pb in ((0, kx, bk, la.k_cache, lb.k_cache), (1, vx, bv, la.v_cache, lb.v_cache)):
            ha, hb = pa.cpu().numpy(), pb.cpu().numpy()
            c32, b32 = ocb.codebook_fp32(D, bits)
            fa = page_fields(la, which, ha)
            for h in range(Hkv):
                idx, gamma, y = oq.quantize(oq.bf16_bits_to_f64(x[:, h]), pi, c32, b32)
                codes, g = slot_fields(fa, slots, h)[:2]
                ok, _ = tie_band_ok(y, codes, idx, b32, 1e-5)
                assert ok, "code mismatch outside the tie band"
                same = np.all(codes == idx, axis=-1)
                assert np.all(np.abs(g[same] - gamma[same]) <= 2e-6 * np.abs(gamma[same]) + 1e-30)
            pb_bytes = ha.reshape(nb, Hkv, -1).shape[-1]
            mask = np.ones((nb, Hkv, pb_bytes), bool)
            from oracle import pack as opack
            rb = opack.page_bytes(D, bits)
            assert rb == pb_bytes
            for s_ in appended:  # the new tokens' records and gammas in every head's page
                blk, off = s_ // 16, s_ % 16
                mask[blk, :, off * 16 * bits:(off + 1) * 16 * bits] = False
                mask[blk, :, 16 * 16 * bits + 4 * off:16 * 16 * bits + 4 * off + 4] = False
            assert np.array_equal(ha.reshape(nb, Hkv, -1)[mask], hb.reshape(nb, Hkv, -1)[mask])
        # the output against the oracle's attention over this cache
        kp, vp = la.k_cache.cpu().numpy(), la.v_cache.cpu().numpy()
        qx = oq.bf16_bits_to_f64(workloads.queries(40 + step, B, Hq, D))
        ref = oa.decode_packed(qx, kp, vp, oracle_layer(la), nb, Hkv, bt, pos + 1, 1 / math.sqrt(D))
        assert_close(out_a.cpu().numpy(), ref, TOL_BF16, pos + 1)
