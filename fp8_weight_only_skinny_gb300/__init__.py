"""Weight-only skinny linear layers (NVFP4 / FP8-E4M3 weights, FP16 activations,
M = 1..8 rows) for GB300, as hand-written sm_103a CUDA kernels behind a C ABI.

The Python surface is a thin ctypes binding with the C names; see
include/skinny.h for the contract of each call.
"""
from ._binding import (  # noqa: F401
    EXPORTS,
    LIB_PATH,
    SK_ERR_CUDA,
    SK_ERR_INVALID_ARG,
    SK_ERR_MISALIGNED,
    SK_ERR_NOT_INITIALIZED,
    SK_ERR_TIMEOUT,
    SK_ERR_UNSUPPORTED_SHAPE,
    SK_ERR_WORKSPACE,
    SK_OK,
    STATUS,
    VARIANT_AUTO,
    VARIANT_SIMT,
    VARIANT_TENSOR,
    SkinnyError,
    fp8_gemm,
    fp8_quantize,
    init,
    last_device_error,
    lib,
    lm_head_argmax,
    lm_head_sample,
    lm_head_verify,
    nvfp4_gemm,
    nvfp4_quantize,
    set_pdl,
    set_variant,
    shutdown,
    status_string,
    stream_workspace,
)
