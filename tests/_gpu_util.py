"""Shared helpers of the GPU parity tests: oracle views of a libtq Layer and
the comparison metrics.  No method arithmetic lives here: the oracle side is
computed by oracle/, the GPU side by libtq."""
import numpy as np

from oracle import attention as oa, codebook as ocb, pack as opack, rotation as orot, rng as orng

D = 128


def oracle_pi(layer):
    """The oracle's own rotation for a Layer's (kind, seed, layer)."""
    if layer.explicit_rotation is not None:
        if layer.rot_kind == orng.KIND_HADAMARD:
            return orot.hadamard_rotation(np.asarray(layer.explicit_rotation, np.float64))
        return np.asarray(layer.explicit_rotation, np.float64)
    return orot.rotation_seeded(layer.rot_kind, layer.seed, layer.layer_index, D)


def oracle_layer(layer):
    cbk = ocb.codebook_fp32(D, layer.bits_k)[0]
    cbv = ocb.codebook_fp32(D, layer.bits_v)[0]
    s = orot.qjl_matrix_seeded(layer.qjl_seed, D, D) if layer.qjl else None
    return oa.PackedLayer(oracle_pi(layer), cbk, cbv, layer.bits_k, layer.bits_v, s)


def pools_host(layer):
    return layer.k_cache.cpu().numpy(), layer.v_cache.cpu().numpy()


def page_fields(layer, which, pool_host):
    bits = layer.bits_k if which == 0 else layer.bits_v
    qjl = layer.qjl and which == 0
    pb = opack.page_bytes(D, bits, qjl)
    pages = opack.pool_pages(pool_host, layer.num_blocks, layer.num_kv_heads, pb)
    return opack.split_pages(pages, D, bits, qjl)


def slot_fields(fields, slots, head):
    """Per-slot rows of split_pages output for one head."""
    slots = np.asarray(slots, np.int64)
    b, t = slots // 16, slots % 16
    return tuple(f[b, head, t] for f in fields)


def max_rel_err(out, ref):
    """max over rows of ||o - o_ref||_inf / ||o_ref||_inf."""
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.max(np.abs(out - ref), axis=-1)
    den = np.max(np.abs(ref), axis=-1)
    return float(np.max(num / np.where(den > 0, den, 1.0)))


def tie_band_ok(y_oracle, idx_gpu, idx_oracle, boundaries, tau):
    """Every code mismatch must sit within tau of the boundary between the codes."""
    y = np.asarray(y_oracle, np.float64)
    mism = idx_gpu != idx_oracle
    if not mism.any():
        return True, 0.0
    lo = np.minimum(idx_gpu, idx_oracle)[mism]
    hi = np.maximum(idx_gpu, idx_oracle)[mism]
    if np.any(hi - lo != 1):
        return False, float(mism.mean())
    beta = np.asarray(boundaries, np.float64)[lo]
    return bool(np.all(np.abs(y[mism] - beta) <= tau)), float(mism.mean())
