"""tq_decode_attention_static: decode attention for callers that cannot allocate.

Some callers of libtq are handed only their input and output buffers -- a
plugin inside a host application that owns all device memory, or a serving
loop that must not call cudaMalloc/cudaFree once running -- and so cannot pass
the workspace tq_decode_attention needs.  This entry point uses a scratch array
inside the library instead.  These tests call it through the C ABI and check
it against tq_decode_attention (caller-provided workspace) on two calls in a
row with different shapes, and that oversized requests are rejected.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes
import math

import numpy as np
import pytest

import workloads
from tests._gpu_util import D, max_rel_err

pytestmark = pytest.mark.gpu

def static_fn(tq):
    fn = tq.lib().tq_decode_attention_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(tq.CacheDesc), ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_int,
                   ctypes.c_int, ctypes.c_void_p]
    return fn


def make_case(cuda, tq, B, Hq, Hkv, ctx, seed, **fmt):
    ctx = np.asarray(ctx, np.int32)
    mb = int(math.ceil(ctx.max() / 16))
    bt, nb = workloads.shuffled_block_table(seed, B, mb)
    layer = tq.Layer(nb, Hkv, seed=seed, layer=1, **fmt)
    kb, vb = workloads.lognormal_channel_kv(seed, B * mb * 16, Hkv, D)
    slots = workloads.prefill_slots(bt, mb * 16)
    dev = lambda a: cuda.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(cuda.bfloat16)
    layer.append(dev(kb), dev(vb), cuda.from_numpy(slots).cuda())
    q = dev(workloads.queries(seed + 1, B, Hq, D))
    return layer, q, cuda.from_numpy(bt).cuda(), cuda.from_numpy(ctx).cuda()


def call_static(cuda, tq, fn, layer, q, bt, ctx, num_splits):
    out = cuda.empty(q.shape, dtype=cuda.float32, device=q.device)
    st = cuda.cuda.current_stream().cuda_stream
    rc = fn(ctypes.byref(layer.desc), ctypes.c_void_p(q.data_ptr()), tq.TQ_BF16, q.shape[0], q.shape[1],
            ctypes.c_void_p(bt.data_ptr()), bt.shape[1], ctypes.c_void_p(ctx.data_ptr()),
            ctypes.c_float(1 / math.sqrt(D)), ctypes.c_void_p(out.data_ptr()), tq.TQ_F32, num_splits,
            ctypes.c_void_p(st))
    return rc, out


def test_static_scratch_matches_workspace_decode_twice(cuda, tqlib):
    """Two calls in a row with different shapes, each equal to the workspace
    call.  Both run the same kernels with the same split count and a fixed merge
    order, so the outputs must agree bit for bit; a stale partial or counter
    left in the shared array by the first call would show up in the second."""
    tq = tqlib
    fn = static_fn(tq)
    cases = [(3, 8, 2, [700, 33, 1024], 5, 0, {}), (2, 32, 4, [2000, 517], 9, 7, {}),
             # a QJL-key layer: the separate query pass runs with the static array as its workspace
             (2, 16, 4, [900, 1500], 13, 0, {"bits_k": 2, "qjl": True})]
    for B, Hq, Hkv, ctx, seed, splits, fmt in cases:
        layer, q, bt, ctxd = make_case(cuda, tq, B, Hq, Hkv, ctx, seed, **fmt)
        ref = layer.decode(q, bt, ctxd, sm_scale=1 / math.sqrt(D), out_dtype=cuda.float32, num_splits=splits)
        rc, out = call_static(cuda, tq, fn, layer, q, bt, ctxd, splits)
        assert rc == tq.TQ_OK, tq.last_error()
        cuda.cuda.synchronize()
        assert tq.get_device_status() == 0
        o, r = out.cpu().numpy(), ref.cpu().numpy()
        assert np.array_equal(o, r), max_rel_err(o, r)


def test_static_scratch_rejects_oversized_requests(cuda, tqlib):
    tq = tqlib
    fn = static_fn(tq)
    layer, q, bt, ctxd = make_case(cuda, tq, 1, 8, 2, [64], 3)
    # 64 sequences x 64 query heads x 64 splits of fp32 partials is far beyond the static scratch
    big_q = cuda.zeros((64, 64, D), dtype=cuda.bfloat16, device="cuda")
    big_bt = cuda.zeros((64, 256), dtype=cuda.int32, device="cuda")
    big_ctx = cuda.zeros((64,), dtype=cuda.int32, device="cuda")
    rc, _ = call_static(cuda, tq, fn, layer, big_q, big_bt, big_ctx, 64)
    assert rc == tq.TQ_ERR_WORKSPACE
    assert "static scratch" in tq.last_error()
