"""ctypes binding of libskinny (include/skinny.h): argument marshalling only.

Every computation runs in the CUDA kernels of libskinny.so.  There is no CPU
or PyTorch fallback: if the library is missing or fails to load, importing the
package raises.  PyTorch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libskinny.so")

STATUS = {
    0: "SK_OK",
    1: "SK_ERR_INVALID_ARG",
    2: "SK_ERR_UNSUPPORTED_SHAPE",
    3: "SK_ERR_MISALIGNED",
    4: "SK_ERR_NOT_INITIALIZED",
    5: "SK_ERR_CUDA",
    6: "SK_ERR_TIMEOUT",
    7: "SK_ERR_WORKSPACE",
}
SK_OK = 0
SK_ERR_INVALID_ARG, SK_ERR_UNSUPPORTED_SHAPE, SK_ERR_MISALIGNED = 1, 2, 3
SK_ERR_NOT_INITIALIZED, SK_ERR_CUDA, SK_ERR_TIMEOUT, SK_ERR_WORKSPACE = 4, 5, 6, 7


class SkinnyError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lib.sk_status_string(status).decode()} ({status})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(LIB_PATH)
    p, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sig = {
        "sk_init": ([ctypes.c_size_t], i),
        "sk_shutdown": ([], i),
        "sk_stream_workspace": ([p, ctypes.c_size_t], i),
        "nvfp4_gemm": ([p, p, p, f, p, i, i, i, p], i),
        "nvfp4_gemm_f16out": ([p, p, p, f, p, i, i, i, p], i),
        "fp8_gemm": ([p, p, p, p, i, i, i, p], i),
        "fp8_gemm_f16out": ([p, p, p, p, i, i, i, p], i),
        "lm_head_argmax": ([p, p, p, f, p, p, i, i, i, p], i),
        "lm_head_verify": ([p, p, p, f, p, p, p, p, i, i, i, p], i),
        "fp8_quantize": ([p, p, p, i, i, p], i),
        "lm_head_sample": ([p, p, p, f, p, p, f, i, f, p, i, i, i, p], i),
        "nvfp4_quantize": ([p, p, p, p, i, i, p], i),
        "sk_status_string": ([i], ctypes.c_char_p),
        "sk_last_device_error": ([p], i),
        "sk_set_pdl": ([i], i),
        "sk_set_variant": ([i], i),
        "sk_version": ([], i),
        "sk_inject_wait_timeout": ([i], None),
        "nvfp4_gemm_noalloc": ([p, p, p, f, p, i, i, i, p], i),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    return L


lib = _load()

# Names declared in include/skinny.h (the tests check that each is exported).
EXPORTS = ("sk_init", "sk_shutdown", "sk_stream_workspace", "nvfp4_gemm", "nvfp4_gemm_f16out", "fp8_gemm",
           "fp8_gemm_f16out", "lm_head_argmax", "lm_head_verify", "lm_head_sample", "fp8_quantize",
           "nvfp4_quantize",
           "sk_status_string", "sk_last_device_error",
           "sk_set_pdl", "sk_set_variant", "sk_inject_wait_timeout", "nvfp4_gemm_noalloc", "sk_version")


def _check(status: int, what: str) -> None:
    if status != SK_OK:
        raise SkinnyError(status, what)


def status_string(status: int) -> str:
    return lib.sk_status_string(int(status)).decode()


def init(workspace_bytes: int = 0) -> None:
    """sk_init on the current CUDA device (call once per device, before graph capture)."""
    _check(lib.sk_init(int(workspace_bytes)), "sk_init")


def shutdown() -> None:
    _check(lib.sk_shutdown(), "sk_shutdown")


def stream_workspace(stream, workspace_bytes: int = 64 << 20) -> None:
    """sk_stream_workspace: a workspace of its own for `stream` (a torch CUDA
    stream) on the current device; 0 bytes removes it."""
    _check(lib.sk_stream_workspace(_stream_ptr(stream), int(workspace_bytes)), "sk_stream_workspace")


def set_pdl(enable: bool) -> bool:
    return bool(lib.sk_set_pdl(1 if enable else 0))


VARIANT_AUTO, VARIANT_TENSOR, VARIANT_SIMT = 0, 1, 2


def set_variant(variant: int) -> int:
    """Kernel variant (VARIANT_AUTO, VARIANT_TENSOR or VARIANT_SIMT); returns the previous one."""
    prev = int(lib.sk_set_variant(int(variant)))
    if prev < 0:
        raise ValueError(f"unknown kernel variant {variant}")
    return prev


def _stream_ptr(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def last_device_error(stream=None) -> int:
    """Synchronise `stream`; return the status of the device error word (and clear it)."""
    return int(lib.sk_last_device_error(_stream_ptr(stream)))


def _dims(x, codes, nv: bool):
    import torch

    if x.dtype != torch.float16 or x.dim() != 2 or not x.is_cuda:
        raise TypeError("x must be a 2-D CUDA float16 tensor [M][K]")
    if codes.dtype != torch.uint8 or codes.dim() != 2 or not codes.is_cuda:
        raise TypeError("W_codes must be a 2-D CUDA uint8 tensor")
    for t in (x, codes):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    M, K = x.shape
    N = codes.shape[0]
    if codes.shape[1] != (K // 2 if nv else K):
        raise ValueError(f"W_codes has shape {tuple(codes.shape)}, expected [N][{K // 2 if nv else K}]")
    return int(M), int(N), int(K)


def nvfp4_gemm(x, W_codes, W_scales, W_gscale: float, y=None, f16_out: bool = False, stream=None):
    """y[M][N] = x . dequant(W)^T for NVFP4 weights (FP32 output, or FP16 with f16_out)."""
    import torch

    M, N, K = _dims(x, W_codes, True)
    if W_scales.dtype != torch.uint8 or tuple(W_scales.shape) != (N, K // 16) or not W_scales.is_contiguous():
        raise ValueError("W_scales must be a contiguous uint8 tensor [N][K/16]")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16 if f16_out else torch.float32, device=x.device)
    fn = lib.nvfp4_gemm_f16out if f16_out else lib.nvfp4_gemm
    _check(fn(x.data_ptr(), W_codes.data_ptr(), W_scales.data_ptr(), float(W_gscale), y.data_ptr(),
              M, N, K, _stream_ptr(stream)), "nvfp4_gemm")
    return y


def fp8_gemm(x, W_codes, W_scales, y=None, f16_out: bool = False, stream=None):
    """y[M][N] = x . dequant(W)^T for FP8-E4M3 weights with 128x128 FP32 block scales."""
    import torch

    M, N, K = _dims(x, W_codes, False)
    if W_scales.dtype != torch.float32 or tuple(W_scales.shape) != ((N + 127) // 128, (K + 127) // 128) \
            or not W_scales.is_contiguous():
        raise ValueError("W_scales must be a contiguous float32 tensor [ceil(N/128)][ceil(K/128)]")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16 if f16_out else torch.float32, device=x.device)
    fn = lib.fp8_gemm_f16out if f16_out else lib.fp8_gemm
    _check(fn(x.data_ptr(), W_codes.data_ptr(), W_scales.data_ptr(), y.data_ptr(), M, N, K,
              _stream_ptr(stream)), "fp8_gemm")
    return y


def lm_head_argmax(x, W_codes, W_scales, W_gscale: float, logits=None, argmax=None,
                   want_logits: bool = True, stream=None):
    """NVFP4 vocabulary projection with the fused per-row argmax.

    Returns (logits or None, argmax int32 [M])."""
    import torch

    M, N, K = _dims(x, W_codes, True)
    if W_scales.dtype != torch.uint8 or tuple(W_scales.shape) != (N, K // 16) or not W_scales.is_contiguous():
        raise ValueError("W_scales must be a contiguous uint8 tensor [N][K/16]")
    if logits is None and want_logits:
        logits = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if argmax is None:
        argmax = torch.empty((M,), dtype=torch.int32, device=x.device)
    _check(lib.lm_head_argmax(x.data_ptr(), W_codes.data_ptr(), W_scales.data_ptr(), float(W_gscale),
                              logits.data_ptr() if logits is not None else None, argmax.data_ptr(),
                              M, N, K, _stream_ptr(stream)), "lm_head_argmax")
    return logits, argmax


def lm_head_verify(x, W_codes, W_scales, W_gscale: float, draft, logits=None, argmax=None, accept=None,
                   want_logits: bool = True, stream=None):
    """lm_head_argmax plus the greedy verification of a speculative round:
    draft is int32 [M - 1] on the device (ignored when M == 1).

    Returns (logits or None, argmax int32 [M], accept int32 [2] = (accepted drafts, bonus token))."""
    import torch

    M, N, K = _dims(x, W_codes, True)
    if W_scales.dtype != torch.uint8 or tuple(W_scales.shape) != (N, K // 16) or not W_scales.is_contiguous():
        raise ValueError("W_scales must be a contiguous uint8 tensor [N][K/16]")
    if M > 1 and (draft is None or draft.dtype != torch.int32 or not draft.is_cuda or draft.numel() < M - 1
                  or not draft.is_contiguous()):
        raise ValueError("draft must be a contiguous CUDA int32 tensor of at least M - 1 tokens")
    if logits is None and want_logits:
        logits = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if argmax is None:
        argmax = torch.empty((M,), dtype=torch.int32, device=x.device)
    if accept is None:
        accept = torch.empty((2,), dtype=torch.int32, device=x.device)
    _check(lib.lm_head_verify(x.data_ptr(), W_codes.data_ptr(), W_scales.data_ptr(), float(W_gscale),
                              logits.data_ptr() if logits is not None else None, argmax.data_ptr(),
                              draft.data_ptr() if (draft is not None and M > 1) else None, accept.data_ptr(),
                              M, N, K, _stream_ptr(stream)), "lm_head_verify")
    return logits, argmax, accept


def _weights_f16(w):
    import torch

    if w.dtype != torch.float16 or w.dim() != 2 or not w.is_cuda or not w.is_contiguous():
        raise TypeError("w must be a contiguous 2-D CUDA float16 tensor [N][K]")
    return int(w.shape[0]), int(w.shape[1])


def fp8_quantize(w, stream=None):
    """FP16 [N][K] -> (codes uint8 [N][K], scales float32 [ceil(N/128)][ceil(K/128)])."""
    import torch

    N, K = _weights_f16(w)
    codes = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    scales = torch.empty(((N + 127) // 128, (K + 127) // 128), dtype=torch.float32, device=w.device)
    _check(lib.fp8_quantize(w.data_ptr(), codes.data_ptr(), scales.data_ptr(), N, K, _stream_ptr(stream)),
           "fp8_quantize")
    return codes, scales


def nvfp4_quantize(w, stream=None):
    """FP16 [N][K] -> (codes uint8 [N][K/2], scales uint8 [N][K/16], tensor scale float32 [1], on the device)."""
    import torch

    N, K = _weights_f16(w)
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((N, K // 16), dtype=torch.uint8, device=w.device)
    gscale = torch.empty((1,), dtype=torch.float32, device=w.device)
    _check(lib.nvfp4_quantize(w.data_ptr(), codes.data_ptr(), scales.data_ptr(), gscale.data_ptr(), N, K,
                              _stream_ptr(stream)), "nvfp4_quantize")
    return codes, scales, gscale


def lm_head_sample(x, W_codes, W_scales, W_gscale: float, u, temperature: float, top_k: int, top_p: float,
                   logits=None, token=None, stream=None):
    """NVFP4 vocabulary projection with a sampled pick per row (temperature /
    top-k / top-p; u is a float32 CUDA tensor of M uniforms in [0, 1)).

    Returns (logits float32 [M][N], token int32 [M])."""
    import torch

    M, N, K = _dims(x, W_codes, True)
    if W_scales.dtype != torch.uint8 or tuple(W_scales.shape) != (N, K // 16) or not W_scales.is_contiguous():
        raise ValueError("W_scales must be a contiguous uint8 tensor [N][K/16]")
    if u.dtype != torch.float32 or not u.is_cuda or u.numel() < M or not u.is_contiguous():
        raise ValueError("u must be a contiguous CUDA float32 tensor of at least M uniforms")
    if logits is None:
        logits = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if token is None:
        token = torch.empty((M,), dtype=torch.int32, device=x.device)
    _check(lib.lm_head_sample(x.data_ptr(), W_codes.data_ptr(), W_scales.data_ptr(), float(W_gscale),
                              logits.data_ptr(), u.data_ptr(), float(temperature), int(top_k), float(top_p),
                              token.data_ptr(), M, N, K, _stream_ptr(stream)), "lm_head_sample")
    return logits, token
