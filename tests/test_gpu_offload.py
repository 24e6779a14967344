"""GPU: offload / restore of cache blocks (byte-exact images, T(Q(X)) = Q(X))."""
import ctypes
import math

import numpy as np
import pytest

import workloads
from oracle import offload as ooff
from tests._gpu_util import D

pytestmark = pytest.mark.gpu


def fmt_tuple(layer):
    f = layer.desc.fmt
    return (f.kv_format, f.bits_k, f.bits_v, f.qjl_k, f.rot_kind, f.norm_mode)


def oracle_image(layer, blocks):
    d = layer.desc
    h = ooff.header(fmt_tuple(layer), D, layer.num_kv_heads, 16, len(blocks),
                    ooff.codebook_hash(d.centroids_k, d.boundaries_k, d.centroids_v, d.boundaries_v))
    return ooff.build_image(layer.k_cache.cpu().numpy(), layer.v_cache.cpu().numpy(), layer.num_blocks,
                            layer.num_kv_heads, layer.page_bytes_k, layer.page_bytes_v, blocks, h)


def filled_layer(cuda, tq, kv, B=3, Hkv=4, T=200, seed=0):
    mb = -(-T // 16)
    bt, nb = workloads.shuffled_block_table(seed + 3, B, mb, num_blocks=B * mb + 5)
    kw = {"packed": dict(), "qjl": dict(bits_k=2, qjl=True, qjl_seed=4), "bf16": dict(kv_format="bf16"),
          "k8v4": dict(kv_format="k8v4", bits_v=3), "polar": dict(kv_format="polar", bits_k=4, bits_v=3)}[kv]
    layer = tq.Layer(nb, Hkv, seed=seed + 1, layer=2, fill=0x11, **kw)
    kb, vb = workloads.scaled_gaussian_kv(seed + 5, B * T, Hkv, D, scale=3.0)
    k = cuda.from_numpy(kb.view(np.int16)).cuda().view(cuda.bfloat16)
    v = cuda.from_numpy(vb.view(np.int16)).cuda().view(cuda.bfloat16)
    layer.append(k, v, cuda.from_numpy(workloads.prefill_slots(bt, T)).cuda())
    return layer, bt, nb, np.full(B, T, np.int32)


def decode(cuda, layer, bt, ctx, q):
    return layer.decode(q, cuda.from_numpy(bt).cuda(), cuda.from_numpy(ctx).cuda(), out_dtype=cuda.float32).cpu().numpy()


@pytest.mark.parametrize("kv", ["packed", "qjl", "bf16", "k8v4", "polar"])
def test_offload_restore_round_trip(cuda, tqlib, kv):
    tq = tqlib
    layer, bt, nb, ctx = filled_layer(cuda, tq, kv)
    q = cuda.from_numpy(workloads.queries(7, bt.shape[0], 8, D).view(np.int16)).cuda().view(cuda.bfloat16)
    ref = decode(cuda, layer, bt, ctx, q)
    blocks = bt.reshape(-1)  # every block in use, in table order (few runs)
    image = layer.offload(blocks)
    cuda.cuda.synchronize()
    assert np.array_equal(image.numpy(), oracle_image(layer, blocks))
    before_k, before_v = layer.k_cache.cpu().numpy(), layer.v_cache.cpu().numpy()
    layer.k_cache.fill_(0xA5)
    layer.v_cache.fill_(0xA5)
    part = blocks[::2]  # restore every other block: the rest stays 0xA5
    layer.restore(part, ooff_slice(image, layer, blocks, part))
    cuda.cuda.synchronize()
    k_now = layer.k_cache.cpu().numpy().reshape(nb, -1)
    v_now = layer.v_cache.cpu().numpy().reshape(nb, -1)
    restored = np.zeros(nb, bool)
    restored[part] = True
    assert np.array_equal(k_now[restored], before_k.reshape(nb, -1)[restored])
    assert np.array_equal(v_now[restored], before_v.reshape(nb, -1)[restored])
    assert np.all(k_now[~restored] == 0xA5) and np.all(v_now[~restored] == 0xA5)
    layer.restore(blocks, image)  # all of them back
    cuda.cuda.synchronize()
    assert np.array_equal(layer.k_cache.cpu().numpy(), np.where(np.isin(np.arange(nb), blocks)[:, None],
                                                                 before_k.reshape(nb, -1), 0xA5).reshape(-1))
    assert np.array_equal(decode(cuda, layer, bt, ctx, q), ref)
    assert tq.get_device_status() == 0


def ooff_slice(image, layer, blocks, part):
    """A pinned image of the `part` blocks cut out of the image of `blocks` (host side)."""
    torch = pytest.importorskip("torch")
    pos = {int(b): i for i, b in enumerate(blocks)}
    kpages, vpages = ooff.image_pages(image.numpy(), layer.num_kv_heads, layer.page_bytes_k, layer.page_bytes_v)
    hdr = bytearray(image.numpy()[: ooff.HEADER].tobytes())
    hdr[48:56] = int(len(part)).to_bytes(8, "little")
    idx = [pos[int(b)] for b in part]
    body = np.concatenate([np.frombuffer(bytes(hdr), np.uint8), kpages[idx].reshape(-1), vpages[idx].reshape(-1)])
    out = torch.empty(body.size, dtype=torch.uint8, pin_memory=True)
    out.copy_(torch.from_numpy(body))
    return out


def test_restore_into_other_blocks(cuda, tqlib):
    """Blocks restored to other physical blocks under a remapped table decode the same."""
    tq = tqlib
    layer, bt, nb, ctx = filled_layer(cuda, tq, "packed", seed=4)
    q = cuda.from_numpy(workloads.queries(9, bt.shape[0], 8, D).view(np.int16)).cuda().view(cuda.bfloat16)
    ref = decode(cuda, layer, bt, ctx, q)
    blocks = bt.reshape(-1)
    image = layer.offload(blocks)
    perm = np.random.default_rng(2).permutation(nb)[: blocks.size].astype(np.int32)  # new homes
    layer.k_cache.fill_(0)
    layer.v_cache.fill_(0)
    layer.restore(perm, image)
    cuda.cuda.synchronize()
    assert np.array_equal(decode(cuda, layer, perm.reshape(bt.shape), ctx, q), ref)


def test_restore_checks_the_header(cuda, tqlib):
    tq = tqlib
    layer, bt, nb, ctx = filled_layer(cuda, tq, "packed", seed=6)
    blocks = bt.reshape(-1)[:5]
    image = layer.offload(blocks)
    cuda.cuda.synchronize()
    other = tq.Layer(nb, layer.num_kv_heads, bits_k=3, seed=1, layer=2)  # another format
    with pytest.raises(tq.TQError, match="another layer format"):
        other.restore(blocks, image)
    with pytest.raises(tq.TQError, match="blocks"):
        layer.restore(blocks[:4], image)
    bad = image.clone().pin_memory()
    bad[8] = 99  # version
    with pytest.raises(tq.TQError) as e:
        layer.restore(blocks, bad)
    assert e.value.status == tq.TQ_ERR_VERSION
    bad = image.clone().pin_memory()
    bad[60] ^= 1  # codebook hash
    with pytest.raises(tq.TQError, match="codebooks"):
        layer.restore(blocks, bad)
    pageable = image.clone()  # not pinned: the device cannot address it
    with pytest.raises(tq.TQError, match="pinned"):
        layer.restore(blocks, pageable)
    with pytest.raises(tq.TQError, match="outside"):
        layer.restore(np.array([0, 1, 2, 3, nb], np.int32), image)
