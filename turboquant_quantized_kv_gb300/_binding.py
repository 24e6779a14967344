"""ctypes binding of libtq (include/tq.h).  Argument marshalling only.

Every computation runs in libtq's CUDA kernels; PyTorch provides device memory
and the current stream.  There is no fallback: if libtq.so is missing or fails
to load, every call raises.
"""

import ctypes
import math
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtq.so")

# ---------------------------------------------------------------- constants
TQ_FORMAT_VERSION = 1
TQ_BLOCK_SIZE = 16
TQ_HEAD_DIM = 128
TQ_MAX_GROUP = 8

TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_WORKSPACE, TQ_ERR_CUDA, TQ_ERR_DEVICE, TQ_ERR_VERSION = range(7)
TQ_F32, TQ_BF16 = 0, 1
TQ_ROT_HADAMARD, TQ_ROT_DENSE, TQ_RNG_QJL = 1, 2, 3
TQ_KV_PACKED, TQ_KV_BF16, TQ_KV_K8V4, TQ_KV_POLAR = 0, 1, 2, 3
TQ_NORM_CORRECTED, TQ_NORM_RAW = 0, 1
TQ_DEV_BAD_SLOT, TQ_DEV_BAD_BLOCK, TQ_DEV_BAD_CONTEXT, TQ_DEV_WAIT_TIMEOUT = 1, 2, 4, 8

STATUS_NAMES = {
    TQ_OK: "TQ_OK", TQ_ERR_INVALID_ARG: "TQ_ERR_INVALID_ARG", TQ_ERR_UNSUPPORTED: "TQ_ERR_UNSUPPORTED",
    TQ_ERR_WORKSPACE: "TQ_ERR_WORKSPACE", TQ_ERR_CUDA: "TQ_ERR_CUDA", TQ_ERR_DEVICE: "TQ_ERR_DEVICE",
    TQ_ERR_VERSION: "TQ_ERR_VERSION",
}


class TQError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


class LayerFormat(ctypes.Structure):
    _fields_ = [("kv_format", ctypes.c_int32), ("bits_k", ctypes.c_int32), ("bits_v", ctypes.c_int32),
                ("qjl_k", ctypes.c_int32), ("rot_kind", ctypes.c_int32), ("norm_mode", ctypes.c_int32)]


class CacheDesc(ctypes.Structure):
    _fields_ = [("format_version", ctypes.c_uint32), ("head_dim", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int64),
                ("fmt", LayerFormat), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("rotation", ctypes.c_void_p), ("qjl_proj", ctypes.c_void_p),
                ("centroids_k", ctypes.c_float * 16), ("boundaries_k", ctypes.c_float * 15),
                ("centroids_v", ctypes.c_float * 16), ("boundaries_v", ctypes.c_float * 15)]


_P = ctypes.POINTER
_D = ctypes.POINTER(CacheDesc)
_SIGNATURES = {
    "tq_make_codebook": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _P(ctypes.c_float), _P(ctypes.c_float)]),
    "tq_make_rotation": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_int, _P(ctypes.c_float)]),
    "tq_page_bytes": (ctypes.c_size_t, [_D, ctypes.c_int]),
    "tq_quantize_append": (ctypes.c_int, [_D, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                          ctypes.c_int64, ctypes.c_void_p]),
    "tq_quantize_append_layers": (ctypes.c_int, [_P(_D), ctypes.c_int, _P(ctypes.c_void_p), _P(ctypes.c_void_p),
                                                 ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]),
    "tq_quantize_rotated": (ctypes.c_int, [_D, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_int64, ctypes.c_void_p]),
    "tq_auto_splits": (ctypes.c_int, [_D, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "tq_workspace_bytes": (ctypes.c_size_t, [_D, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "tq_decode_attention": (ctypes.c_int, [_D, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_float,
                                           ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                           ctypes.c_int, ctypes.c_void_p]),
    "tq_append_decode": (ctypes.c_int, [_D, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_float,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                        ctypes.c_int, ctypes.c_void_p]),
    "tq_decode_step": (ctypes.c_int, [_D, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]),
    "tq_dequantize": (ctypes.c_int, [_D, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                     ctypes.c_int, ctypes.c_void_p]),
    "tq_image_bytes": (ctypes.c_size_t, [_D, ctypes.c_int64]),
    "tq_offload_blocks": (ctypes.c_int, [_D, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t,
                                         ctypes.c_void_p]),
    "tq_restore_blocks": (ctypes.c_int, [_D, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t,
                                         ctypes.c_void_p]),
    "tq_get_device_status": (ctypes.c_int, [ctypes.c_void_p, _P(ctypes.c_int32)]),
    "tq_last_error": (ctypes.c_char_p, []),
    "tq_format_version": (ctypes.c_uint32, []),
    "tq_launch_count": (ctypes.c_uint64, []),
}

_lib = None


def lib():
    """The loaded libtq (raises if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libtq.so is not built (%s); run turboquant_quantized_kv_gb300.build.build()" % LIB_PATH)
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        if handle.tq_format_version() != TQ_FORMAT_VERSION:
            raise RuntimeError("libtq format version mismatch")
        _lib = handle
    return _lib


def last_error():
    return lib().tq_last_error().decode("utf-8", "replace")


def _check(status):
    if status != TQ_OK:
        raise TQError(status, last_error())


# ------------------------------------------------------------------ set-up

def make_codebook(bits, head_dim=TQ_HEAD_DIM):
    """(centroids fp32 [2^bits], boundaries fp32 [2^bits - 1]) from tq_make_codebook."""
    k = 1 << bits
    c = (ctypes.c_float * k)()
    b = (ctypes.c_float * max(k - 1, 1))()
    _check(lib().tq_make_codebook(head_dim, bits, c, b))
    return np.frombuffer(c, dtype=np.float32).copy(), np.frombuffer(b, dtype=np.float32)[: k - 1].copy()


def make_rotation(kind, seed, layer=0, head_dim=TQ_HEAD_DIM):
    """Host fp32 signs [d] (Hadamard) or matrix [d, d] (dense, QJL) from tq_make_rotation."""
    n = head_dim if kind == TQ_ROT_HADAMARD else head_dim * head_dim
    out = (ctypes.c_float * n)()
    _check(lib().tq_make_rotation(kind, head_dim, ctypes.c_uint64(seed), layer, out))
    arr = np.frombuffer(out, dtype=np.float32).copy()
    return arr if kind == TQ_ROT_HADAMARD else arr.reshape(head_dim, head_dim)


# ------------------------------------------------------------ tensor glue

def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return TQ_F32
    if t.dtype == torch.bfloat16:
        return TQ_BF16
    raise TypeError("unsupported dtype %s (float32 or bfloat16)" % t.dtype)


def _ptr(t, name):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class Layer:
    """One layer of the paged cache: device pools, rotation and codebooks.

    kv_format: "packed" (TurboQuant codes), "bf16" (boundary layers), "k8v4"
    (FP8 E4M3 keys with TurboQuant values of bits_v) or "polar" (PolarQuant
    angle codes of bits_k / bits_v bits with an fp16 radius; Hadamard only).
    The descriptor (`desc`) points at tensors owned by this object.
    """

    def __init__(self, num_blocks, num_kv_heads, *, kv_format="packed", bits_k=4, bits_v=4, qjl=False,
                 rot_kind=TQ_ROT_HADAMARD, seed=0, layer=0, qjl_seed=None, norm_mode=TQ_NORM_CORRECTED,
                 device="cuda", rotation=None, qjl_proj=None, fill=0):
        torch = _torch()
        self.num_blocks = int(num_blocks)
        self.num_kv_heads = int(num_kv_heads)
        self.head_dim = TQ_HEAD_DIM
        if kv_format not in ("packed", "bf16", "k8v4", "polar"):
            raise ValueError("kv_format must be 'packed', 'bf16', 'k8v4' or 'polar'")
        self.kv_format = kv_format
        self.packed = kv_format == "packed"
        self.k8v4 = kv_format == "k8v4"
        self.polar = kv_format == "polar"
        coded_v = self.packed or self.k8v4 or self.polar  # rotated, coded layers
        d = CacheDesc()
        d.format_version = TQ_FORMAT_VERSION
        d.head_dim = TQ_HEAD_DIM
        d.num_kv_heads = self.num_kv_heads
        d.block_size = TQ_BLOCK_SIZE
        d.num_blocks = self.num_blocks
        d.fmt.kv_format = {"packed": TQ_KV_PACKED, "bf16": TQ_KV_BF16, "k8v4": TQ_KV_K8V4,
                           "polar": TQ_KV_POLAR}[kv_format]
        if self.k8v4:
            bits_k = 8
        d.fmt.bits_k = bits_k if coded_v else 0
        d.fmt.bits_v = bits_v if coded_v else 0
        d.fmt.qjl_k = 1 if (qjl and self.packed) else 0
        d.fmt.rot_kind = rot_kind if coded_v else 0
        d.fmt.norm_mode = norm_mode
        self.bits_k, self.bits_v, self.qjl, self.rot_kind = bits_k, bits_v, bool(qjl and self.packed), rot_kind
        self.seed, self.layer_index = seed, layer
        self.qjl_seed = seed if qjl_seed is None else qjl_seed
        self.explicit_rotation = rotation
        self.rotation_host = None
        self.qjl_host = None
        self.cb_k = self.cb_v = None
        if coded_v:
            self.cb_k = make_codebook(bits_k) if self.packed else None
            self.cb_v = make_codebook(bits_v) if not self.polar else None
            if self.packed:
                for i, v in enumerate(self.cb_k[0]):
                    d.centroids_k[i] = float(v)
                for i, v in enumerate(self.cb_k[1]):
                    d.boundaries_k[i] = float(v)
            if self.cb_v is not None:
                for i, v in enumerate(self.cb_v[0]):
                    d.centroids_v[i] = float(v)
                for i, v in enumerate(self.cb_v[1]):
                    d.boundaries_v[i] = float(v)
            rot = make_rotation(rot_kind, seed, layer) if rotation is None else np.asarray(rotation, np.float32)
            self.rotation_host = rot
            self.rotation = torch.from_numpy(np.ascontiguousarray(rot)).to(device)
            d.rotation = self.rotation.data_ptr()
            if self.qjl:
                s = make_rotation(TQ_RNG_QJL, seed if qjl_seed is None else qjl_seed) if qjl_proj is None \
                    else np.asarray(qjl_proj, np.float32)
                self.qjl_host = s
                self.qjl_proj = torch.from_numpy(np.ascontiguousarray(s)).to(device)
                d.qjl_proj = self.qjl_proj.data_ptr()
        self.desc = d
        self.page_bytes_k = self.page_bytes(0)
        self.page_bytes_v = self.page_bytes(1)
        nk = self.num_blocks * self.num_kv_heads * self.page_bytes_k
        nv = self.num_blocks * self.num_kv_heads * self.page_bytes_v
        self.k_cache = torch.full((nk,), fill, dtype=torch.uint8, device=device)
        self.v_cache = torch.full((nv,), fill, dtype=torch.uint8, device=device)
        d.k_cache = self.k_cache.data_ptr()
        d.v_cache = self.v_cache.data_ptr()

    def page_bytes(self, which):
        n = lib().tq_page_bytes(ctypes.byref(self.desc), which)
        if n == 0:
            raise TQError(TQ_ERR_INVALID_ARG, last_error() or "invalid descriptor")
        return int(n)

    # -------------------------------------------------------------- calls
    def append(self, k, v, slot_mapping, stream=None):
        """Quantize-on-append of k, v [n_tokens, H_kv, d] into slot_mapping [n_tokens] (int64)."""
        ref = k if k is not None else v
        n = int(ref.shape[0])
        _check(lib().tq_quantize_append(ctypes.byref(self.desc), _ptr(k, "k"), _ptr(v, "v"), _dtype_code(ref),
                                        _ptr(slot_mapping, "slot_mapping"), n, _stream(stream)))

    def quantize_rotated(self, which, y, norms, slot_mapping, stream=None):
        """The quantizer alone on rotated unit coordinates y [n, H_kv, d] (fp32) with norms [n, H_kv]."""
        _check(lib().tq_quantize_rotated(ctypes.byref(self.desc), which, _ptr(y, "y"), _ptr(norms, "norms"),
                                         _ptr(slot_mapping, "slot_mapping"), int(y.shape[0]), _stream(stream)))

    def workspace_bytes(self, batch, num_q_heads, max_blocks_per_seq, num_splits=0):
        n = lib().tq_workspace_bytes(ctypes.byref(self.desc), batch, num_q_heads, max_blocks_per_seq, num_splits)
        if n == 0:
            raise TQError(TQ_ERR_INVALID_ARG, last_error() or "invalid sizes")
        return int(n)

    def auto_splits(self, batch, num_q_heads, max_blocks_per_seq):
        return int(lib().tq_auto_splits(ctypes.byref(self.desc), batch, num_q_heads, max_blocks_per_seq))

    def decode(self, q, block_table, context_lens, sm_scale=None, out=None, out_dtype=None, num_splits=0,
               workspace=None, stream=None):
        """Decode attention.  q [B, H_q, d]; block_table int32 [B, max_blocks]; context_lens int32 [B]."""
        torch = _torch()
        bsz, hq, _ = q.shape
        max_blocks = int(block_table.shape[1])
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.head_dim)
        if out is None:
            out = torch.empty(q.shape, dtype=q.dtype if out_dtype is None else out_dtype, device=q.device)
        if workspace is None:
            workspace = torch.zeros(self.workspace_bytes(bsz, hq, max_blocks, num_splits), dtype=torch.uint8,
                                    device=q.device)
        _check(lib().tq_decode_attention(ctypes.byref(self.desc), _ptr(q, "q"), _dtype_code(q), bsz, hq,
                                         _ptr(block_table, "block_table"), max_blocks,
                                         _ptr(context_lens, "context_lens"), ctypes.c_float(sm_scale),
                                         _ptr(out, "out"), _dtype_code(out), _ptr(workspace, "workspace"),
                                         workspace.numel(), num_splits, _stream(stream)))
        return out

    def append_decode(self, k, v, slot_mapping, q, block_table, context_lens, sm_scale=None, out=None,
                      out_dtype=None, num_splits=0, workspace=None, stream=None):
        """append(k, v, slot_mapping) then decode(q, ...) in one call (tq_append_decode: the
        decode's prologue overlaps the append).  Returns out."""
        torch = _torch()
        ref = k if k is not None else v
        n = int(ref.shape[0]) if ref is not None else 0
        bsz, hq, _ = q.shape
        max_blocks = int(block_table.shape[1])
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.head_dim)
        if out is None:
            out = torch.empty(q.shape, dtype=q.dtype if out_dtype is None else out_dtype, device=q.device)
        if workspace is None:
            workspace = torch.zeros(self.workspace_bytes(bsz, hq, max_blocks, num_splits), dtype=torch.uint8,
                                    device=q.device)
        _check(lib().tq_append_decode(ctypes.byref(self.desc), _ptr(k, "k"), _ptr(v, "v"),
                                      _dtype_code(ref) if ref is not None else TQ_BF16,
                                      _ptr(slot_mapping, "slot_mapping"), n, _ptr(q, "q"), _dtype_code(q), bsz, hq,
                                      _ptr(block_table, "block_table"), max_blocks,
                                      _ptr(context_lens, "context_lens"), ctypes.c_float(sm_scale),
                                      _ptr(out, "out"), _dtype_code(out), _ptr(workspace, "workspace"),
                                      workspace.numel(), num_splits, _stream(stream)))
        return out

    def decode_step(self, k_new, v_new, q, block_table, context_lens, sm_scale=None, out=None, out_dtype=None,
                    num_splits=0, workspace=None, stream=None):
        """One decode step in one kernel (tq_decode_step): k_new, v_new [B, H_kv, d] are the new
        tokens, written at position context_lens[b] - 1 of each sequence (context_lens already
        counts them), then decode(q, ...).  Returns out."""
        torch = _torch()
        bsz, hq, _ = q.shape
        max_blocks = int(block_table.shape[1])
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.head_dim)
        if out is None:
            out = torch.empty(q.shape, dtype=q.dtype if out_dtype is None else out_dtype, device=q.device)
        if workspace is None:
            workspace = torch.zeros(self.workspace_bytes(bsz, hq, max_blocks, num_splits), dtype=torch.uint8,
                                    device=q.device)
        _check(lib().tq_decode_step(ctypes.byref(self.desc), _ptr(k_new, "k_new"), _ptr(v_new, "v_new"),
                                    _dtype_code(k_new), _ptr(q, "q"), _dtype_code(q), bsz, hq,
                                    _ptr(block_table, "block_table"), max_blocks, _ptr(context_lens, "context_lens"),
                                    ctypes.c_float(sm_scale), _ptr(out, "out"), _dtype_code(out),
                                    _ptr(workspace, "workspace"), workspace.numel(), num_splits, _stream(stream)))
        return out

    def image_bytes(self, n_blocks):
        n = lib().tq_image_bytes(ctypes.byref(self.desc), int(n_blocks))
        if n == 0:
            raise TQError(TQ_ERR_INVALID_ARG, last_error() or "invalid descriptor")
        return int(n)

    def offload(self, blocks, image=None, stream=None):
        """Host image (pinned uint8 tensor) of the pages of `blocks` (block ids), see
        tq_offload_blocks.  The image is complete once the stream reaches this call."""
        torch = _torch()
        ids = np.ascontiguousarray(np.asarray(blocks, dtype=np.int32).reshape(-1))
        if image is None:
            image = torch.empty(self.image_bytes(ids.size), dtype=torch.uint8, pin_memory=True)
        if image.is_cuda:
            raise ValueError("image must be a host (pinned) tensor")
        _check(lib().tq_offload_blocks(ctypes.byref(self.desc), ids.ctypes.data_as(ctypes.c_void_p), ids.size,
                                       ctypes.c_void_p(image.data_ptr()), image.numel(), _stream(stream)))
        return image

    def restore(self, blocks, image, stream=None):
        """Copies an image's pages into `blocks` (tq_restore_blocks)."""
        ids = np.ascontiguousarray(np.asarray(blocks, dtype=np.int32).reshape(-1))
        if image.is_cuda:
            raise ValueError("image must be a host (pinned) tensor")
        _check(lib().tq_restore_blocks(ctypes.byref(self.desc), ids.ctypes.data_as(ctypes.c_void_p), ids.size,
                                       ctypes.c_void_p(image.data_ptr()), image.numel(), _stream(stream)))

    def dequantize(self, which, slots, out_dtype=None, stream=None):
        """x_hat [n, H_kv, d] of the K (which=0) or V (which=1) records at slots [n] (int64)."""
        torch = _torch()
        dt = torch.float32 if out_dtype is None else out_dtype
        out = torch.empty((int(slots.shape[0]), self.num_kv_heads, self.head_dim), dtype=dt, device=slots.device)
        _check(lib().tq_dequantize(ctypes.byref(self.desc), which, _ptr(slots, "slots"), int(slots.shape[0]),
                                   _ptr(out, "out"), _dtype_code(out), _stream(stream)))
        return out


def append_layers(layers, ks, vs, slot_mapping, stream=None):
    """Quantize-on-append of the same tokens into several layers (tq_quantize_append_layers):
    ks[l], vs[l] [n_tokens, H_kv, d] are layer l's inputs (either list may be None)."""
    n_layers = len(layers)
    descs = (ctypes.POINTER(CacheDesc) * n_layers)(*[ctypes.pointer(ly.desc) for ly in layers])
    def ptrs(ts, name):
        if ts is None:
            return None
        return (ctypes.c_void_p * n_layers)(*[_ptr(t, name) for t in ts])
    ref = (ks if ks is not None else vs)[0]
    _check(lib().tq_quantize_append_layers(descs, n_layers, ptrs(ks, "k"), ptrs(vs, "v"), _dtype_code(ref),
                                           _ptr(slot_mapping, "slot_mapping"), int(ref.shape[0]), _stream(stream)))


def get_device_status(stream=None):
    """Synchronizes the stream and returns (and clears) the sticky device status bits."""
    code = ctypes.c_int32(0)
    _check(lib().tq_get_device_status(_stream(stream), ctypes.byref(code)))
    return int(code.value)


def launch_count():
    """Kernels libtq has enqueued in this process (a launch captured in a graph counts once)."""
    return int(lib().tq_launch_count())
