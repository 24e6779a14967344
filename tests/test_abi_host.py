"""C-ABI checks that need no GPU: exports, host set-up math against the oracle,
and host-side argument validation (no kernel is launched)."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import codebook as ocb, rng as orng, rotation as orot

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "tq.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(tqlib):
    names = declared_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(tqlib.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_bit_exact_with_oracle(tqlib, bits):
    c, b = tqlib.make_codebook(bits)
    oc, ob = ocb.codebook_fp32(128, bits)
    assert np.array_equal(c.view(np.uint32), oc.view(np.uint32))
    assert np.array_equal(b.view(np.uint32), ob.view(np.uint32))


@pytest.mark.parametrize("seed,layer", [(0, 0), (0, 5), (12345, 31), (2 ** 63 + 7, 2)])
def test_hadamard_signs_match_oracle(tqlib, seed, layer):
    s = tqlib.make_rotation(tqlib.TQ_ROT_HADAMARD, seed, layer)
    assert np.array_equal(s.astype(np.float64), orng.signs(seed, layer, 128))


def test_dense_rotation_and_qjl_match_oracle(tqlib):
    pi = tqlib.make_rotation(tqlib.TQ_ROT_DENSE, 7, 3).astype(np.float64)
    ref = orot.dense_rotation_seeded(7, 3, 128)
    assert np.max(np.abs(pi - ref)) < 1.2e-7  # fp32 rounding of the fp64 Haar Q
    assert np.max(np.abs(pi @ pi.T - np.eye(128))) < 2e-6
    s = tqlib.make_rotation(tqlib.TQ_RNG_QJL, 9).astype(np.float64)
    sref = orot.qjl_matrix_seeded(9, 128, 128)
    assert np.max(np.abs(s - sref) / np.maximum(1.0, np.abs(sref))) < 1e-6


def fake_desc(tq, **kw):
    d = tq.CacheDesc()
    d.format_version = tq.TQ_FORMAT_VERSION
    d.head_dim = 128
    d.num_kv_heads = 8
    d.block_size = 16
    d.num_blocks = 10
    d.fmt.kv_format = tq.TQ_KV_PACKED
    d.fmt.bits_k, d.fmt.bits_v = 4, 4
    d.fmt.rot_kind = tq.TQ_ROT_HADAMARD
    d.k_cache, d.v_cache, d.rotation = 0x10000, 0x20000, 0x30000
    for which in ("k", "v"):
        c, b = tq.make_codebook(getattr(d.fmt, "bits_" + which))
        for i, v in enumerate(c):
            getattr(d, "centroids_" + which)[i] = float(v)
        for i, v in enumerate(b):
            getattr(d, "boundaries_" + which)[i] = float(v)
    for k, v in kw.items():
        if hasattr(d.fmt, k) and k not in ("k_cache",):
            setattr(d.fmt, k, v)
        else:
            setattr(d, k, v)
    return d


def test_page_bytes(tqlib):
    tq = tqlib
    lib = tq.lib()
    d = fake_desc(tq)
    assert lib.tq_page_bytes(ctypes.byref(d), 0) == 1088
    d = fake_desc(tq, bits_k=3)
    # codebook of K must match its bit width: rebuild tables for 3 bits
    c, b = tq.make_codebook(3)
    for i, v in enumerate(c):
        d.centroids_k[i] = float(v)
    for i, v in enumerate(b):
        d.boundaries_k[i] = float(v)
    assert lib.tq_page_bytes(ctypes.byref(d), 0) == 832
    assert lib.tq_page_bytes(ctypes.byref(d), 1) == 1088
    d = fake_desc(tq, kv_format=tq.TQ_KV_BF16)
    assert lib.tq_page_bytes(ctypes.byref(d), 0) == 4096
    assert lib.tq_workspace_bytes(ctypes.byref(fake_desc(tq)), 2, 16, 10, 3) > 2 * 16 * 3 * 128 * 4


def test_descriptor_validation(tqlib):
    tq = tqlib
    lib = tq.lib()

    launches0 = tq.launch_count()

    def status(d):
        return lib.tq_quantize_append(ctypes.byref(d), ctypes.c_void_p(0x1000), None, tq.TQ_F32,
                                      ctypes.c_void_p(0x2000), 4, None)

    assert status(fake_desc(tq, format_version=99)) == tq.TQ_ERR_VERSION
    assert status(fake_desc(tq, head_dim=64)) == tq.TQ_ERR_UNSUPPORTED
    assert status(fake_desc(tq, block_size=32)) == tq.TQ_ERR_UNSUPPORTED
    assert status(fake_desc(tq, k_cache=0x10008)) == tq.TQ_ERR_INVALID_ARG
    assert status(fake_desc(tq, bits_k=5)) == tq.TQ_ERR_INVALID_ARG
    assert status(fake_desc(tq, rot_kind=7)) == tq.TQ_ERR_INVALID_ARG
    assert status(fake_desc(tq, qjl_k=1)) == tq.TQ_ERR_INVALID_ARG  # no projection given
    d = fake_desc(tq)
    d.centroids_k[3] = d.centroids_k[3] * 1.01  # breaks antisymmetry
    assert status(d) == tq.TQ_ERR_INVALID_ARG
    assert "antisymmetric" in tq.last_error()
    d = fake_desc(tq)
    assert lib.tq_quantize_append(ctypes.byref(d), ctypes.c_void_p(0x1000), None, 7, ctypes.c_void_p(0x2000), 4,
                                  None) == tq.TQ_ERR_INVALID_ARG
    assert lib.tq_quantize_append(ctypes.byref(d), ctypes.c_void_p(0x1004), None, tq.TQ_F32,
                                  ctypes.c_void_p(0x2000), 4, None) == tq.TQ_ERR_INVALID_ARG
    assert lib.tq_quantize_append(ctypes.byref(d), None, None, tq.TQ_F32, ctypes.c_void_p(0x2000), 4,
                                  None) == tq.TQ_ERR_INVALID_ARG
    assert lib.tq_quantize_append(ctypes.byref(d), ctypes.c_void_p(0x1000), None, tq.TQ_F32, None, 0,
                                  None) == tq.TQ_OK  # zero tokens: nothing to do
    # decode: head counts and workspace are checked on the host
    ws = ctypes.c_void_p(0x40000)
    assert lib.tq_decode_attention(ctypes.byref(d), ctypes.c_void_p(0x1000), tq.TQ_F32, 2, 12, ctypes.c_void_p(8),
                                   4, ctypes.c_void_p(8), 0.1, ctypes.c_void_p(0x1000), tq.TQ_F32, ws, 1 << 20, 1,
                                   None) == tq.TQ_ERR_INVALID_ARG  # 12 % 8 != 0
    assert lib.tq_decode_attention(ctypes.byref(d), ctypes.c_void_p(0x1000), tq.TQ_F32, 0, 8, None, 4, None, 0.1,
                                   None, tq.TQ_F32, None, 0, 0, None) == tq.TQ_OK  # empty batch
    assert lib.tq_dequantize(ctypes.byref(d), 2, ctypes.c_void_p(8), 1, ctypes.c_void_p(8), tq.TQ_F32,
                             None) == tq.TQ_ERR_INVALID_ARG
    assert tq.launch_count() == launches0  # rejected and empty calls enqueue nothing


def test_append_decode_checks_both_calls_before_launching(tqlib):
    """tq_append_decode checks the append's and the decode's arguments before it
    enqueues anything: an invalid decode part rejects the call with nothing launched."""
    tq = tqlib
    lib = tq.lib()
    d = fake_desc(tq)
    launches0 = tq.launch_count()
    ws = ctypes.c_void_p(0x40000)

    def call(k, n_tokens, hq, batch=2):
        return lib.tq_append_decode(ctypes.byref(d), k, None, tq.TQ_F32, ctypes.c_void_p(0x2000), n_tokens,
                                    ctypes.c_void_p(0x1000), tq.TQ_F32, batch, hq, ctypes.c_void_p(8), 4,
                                    ctypes.c_void_p(8), 0.1, ctypes.c_void_p(0x1000), tq.TQ_F32, ws, 1 << 20, 1, None)

    assert call(ctypes.c_void_p(0x1004), 4, 8) == tq.TQ_ERR_INVALID_ARG  # misaligned k
    assert "tq_append_decode" in tq.last_error() and "aligned" in tq.last_error()
    assert call(ctypes.c_void_p(0x1000), 4, 12) == tq.TQ_ERR_INVALID_ARG  # valid append, 12 % 8 != 0
    assert "num_q_heads" in tq.last_error()
    assert call(ctypes.c_void_p(0x1000), 0, 8, batch=0) == tq.TQ_OK  # nothing to append or decode
    assert tq.launch_count() == launches0


def test_decode_step_checks(tqlib):
    """tq_decode_step takes packed Hadamard layers without QJL keys and checks its new
    tokens before anything is launched (the decode part as tq_decode_attention)."""
    tq = tqlib
    lib = tq.lib()
    launches0 = tq.launch_count()
    ws = ctypes.c_void_p(0x40000)

    def call(d, k, v, hq=8, batch=2, in_dtype=None):
        return lib.tq_decode_step(ctypes.byref(d), k, v, tq.TQ_BF16 if in_dtype is None else in_dtype,
                                  ctypes.c_void_p(0x1000), tq.TQ_F32, batch, hq, ctypes.c_void_p(8), 4,
                                  ctypes.c_void_p(8), 0.1, ctypes.c_void_p(0x1000), tq.TQ_F32, ws, 1 << 20, 1, None)

    good = ctypes.c_void_p(0x2000)
    for kw in (dict(rot_kind=tq.TQ_ROT_DENSE), dict(qjl_k=1, qjl_proj=0x50000), dict(kv_format=tq.TQ_KV_BF16),
               dict(kv_format=tq.TQ_KV_K8V4, bits_k=8)):
        assert call(fake_desc(tq, **kw), good, good) == tq.TQ_ERR_UNSUPPORTED, kw
        assert "tq_decode_step" in tq.last_error()
    d = fake_desc(tq)
    assert call(d, None, good) == tq.TQ_ERR_INVALID_ARG  # null k_new
    assert call(d, good, ctypes.c_void_p(0x2008)) == tq.TQ_ERR_INVALID_ARG  # misaligned v_new
    assert "aligned" in tq.last_error()
    assert call(d, good, good, in_dtype=7) == tq.TQ_ERR_INVALID_ARG  # bad dtype
    assert call(d, good, good, hq=12) == tq.TQ_ERR_INVALID_ARG  # 12 % 8 != 0 (the decode's check)
    assert call(d, good, good, batch=0) == tq.TQ_OK  # nothing to do
    assert tq.launch_count() == launches0


def test_make_args_rejected(tqlib):
    lib = tqlib.lib()
    c = (ctypes.c_float * 16)()
    b = (ctypes.c_float * 15)()
    assert lib.tq_make_codebook(128, 5, c, b) == tqlib.TQ_ERR_INVALID_ARG
    assert lib.tq_make_codebook(128, 2, None, b) == tqlib.TQ_ERR_INVALID_ARG
    out = (ctypes.c_float * 128)()
    assert lib.tq_make_rotation(tqlib.TQ_ROT_HADAMARD, 96, 0, 0, out) == tqlib.TQ_ERR_INVALID_ARG
    assert lib.tq_make_rotation(9, 128, 0, 0, out) == tqlib.TQ_ERR_INVALID_ARG


def test_k8v4_descriptor(tqlib):
    """k8v4 layers: FP8 key pages of 16 x 128 bytes, packed value pages; keys must be
    declared 8-bit, without QJL; the key codebook is not used."""
    tq = tqlib
    lib = tq.lib()
    d = fake_desc(tq, kv_format=tq.TQ_KV_K8V4, bits_k=8)
    for i in range(16):
        d.centroids_k[i] = 0.0  # ignored for FP8 keys
    assert lib.tq_page_bytes(ctypes.byref(d), 0) == 2048
    assert lib.tq_page_bytes(ctypes.byref(d), 1) == 1088
    launches0 = tq.launch_count()

    def append(desc):
        return lib.tq_quantize_append(ctypes.byref(desc), ctypes.c_void_p(0x1000), None, tq.TQ_F32,
                                      ctypes.c_void_p(0x2000), 4, None)

    assert append(fake_desc(tq, kv_format=tq.TQ_KV_K8V4, bits_k=4)) == tq.TQ_ERR_INVALID_ARG
    assert "bits_k" in tq.last_error()
    assert append(fake_desc(tq, kv_format=tq.TQ_KV_K8V4, bits_k=8, qjl_k=1)) == tq.TQ_ERR_INVALID_ARG
    bad = fake_desc(tq, kv_format=tq.TQ_KV_K8V4, bits_k=8)
    bad.centroids_v[2] = bad.centroids_v[2] * 1.5  # breaks the value codebook
    assert append(bad) == tq.TQ_ERR_INVALID_ARG
    assert tq.launch_count() == launches0


def test_polar_descriptor(tqlib):
    """Polar layers: pages of 16 angle-code records + 16 fp16 radii; Hadamard only, no
    QJL, 2..4 bits; the codebook fields are ignored."""
    tq = tqlib
    lib = tq.lib()
    d = fake_desc(tq, kv_format=tq.TQ_KV_POLAR, bits_k=4, bits_v=3)
    for i in range(16):
        d.centroids_k[i] = d.centroids_v[i] = 0.0  # ignored
    assert lib.tq_page_bytes(ctypes.byref(d), 0) == 1056
    assert lib.tq_page_bytes(ctypes.byref(d), 1) == 800
    assert lib.tq_page_bytes(ctypes.byref(fake_desc(tq, kv_format=tq.TQ_KV_POLAR, bits_k=2)), 0) == 544
    launches0 = tq.launch_count()

    def append(desc):
        return lib.tq_quantize_append(ctypes.byref(desc), ctypes.c_void_p(0x1000), None, tq.TQ_F32,
                                      ctypes.c_void_p(0x2000), 4, None)

    assert append(fake_desc(tq, kv_format=tq.TQ_KV_POLAR, rot_kind=tq.TQ_ROT_DENSE)) == tq.TQ_ERR_UNSUPPORTED
    assert append(fake_desc(tq, kv_format=tq.TQ_KV_POLAR, qjl_k=1)) == tq.TQ_ERR_INVALID_ARG
    assert append(fake_desc(tq, kv_format=tq.TQ_KV_POLAR, bits_v=5)) == tq.TQ_ERR_INVALID_ARG
    assert tq.launch_count() == launches0
