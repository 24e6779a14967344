"""TurboQuant quantized KV cache for NVIDIA GB300 (sm_103a).

Python face of libtq (include/tq.h): quantize-on-append into a paged cache of
Lloyd-Max codes with fp32 norm correction (optional 1-bit QJL residual for
keys; a PolarQuant angle-code variant), and decode attention run directly on
the packed cache.  All compute is
in libtq's CUDA kernels; this package only marshals arguments.
"""

from ._binding import (  # noqa: F401
    CacheDesc, Layer, LayerFormat, TQError, append_layers, get_device_status, last_error, launch_count, lib,
    make_codebook,
    make_rotation,
    LIB_PATH, STATUS_NAMES,
    TQ_BF16, TQ_BLOCK_SIZE, TQ_DEV_BAD_BLOCK, TQ_DEV_BAD_CONTEXT, TQ_DEV_BAD_SLOT, TQ_DEV_WAIT_TIMEOUT,
    TQ_ERR_CUDA, TQ_ERR_DEVICE, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_VERSION, TQ_ERR_WORKSPACE,
    TQ_F32, TQ_FORMAT_VERSION, TQ_HEAD_DIM, TQ_KV_BF16, TQ_KV_K8V4, TQ_KV_PACKED, TQ_KV_POLAR, TQ_MAX_GROUP, TQ_NORM_CORRECTED,
    TQ_NORM_RAW, TQ_OK, TQ_RNG_QJL, TQ_ROT_DENSE, TQ_ROT_HADAMARD,
)
