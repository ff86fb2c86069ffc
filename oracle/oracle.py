"""ctypes front end of ``oracle.c`` (test infrastructure only).

The C file holds all of the arithmetic (bit-field decoding of FP16, E2M1 and
E4M3, and the double-precision sums); this module only marshals numpy arrays.
See the header of ``oracle.c`` for what is computed and which passages of the
pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so with gcc (OpenMP on)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", _SRC,
             "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        # SKINNY_ORACLE_LIB lets the mutation tests load a deliberately broken
        # build of oracle.c; normally the library is built from oracle.c here.
        lib = ctypes.CDLL(os.environ.get("SKINNY_ORACLE_LIB") or build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_e2m1_to_f64.restype = ctypes.c_double
        lib.oracle_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_nvfp4_linear.restype = None
        lib.oracle_nvfp4_linear.argtypes = [i64, i64, i64, p, p, p, ctypes.c_float,
                                            p, i64, p, p]
        lib.oracle_fp8_linear.restype = None
        lib.oracle_fp8_linear.argtypes = [i64, i64, i64, p, p, p, p, i64, p, p]
        lib.oracle_argmax_rows.restype = None
        lib.oracle_argmax_rows.argtypes = [i64, i64, p, p]
        lib.oracle_verify.restype = None
        lib.oracle_verify.argtypes = [i64, p, p, p]
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_set_threads.restype = None
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def threads() -> int:
    """OpenMP threads the oracle's column loop uses."""
    return int(_load().oracle_threads())


def set_threads(n: int) -> None:
    """Threads the column loops use from now on (the results do not depend on it)."""
    _load().oracle_set_threads(int(n))


def f16_to_f64(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_f16_to_f64(int(v)) for v in b], dtype=np.float64)


def e2m1_to_f64(codes) -> np.ndarray:
    lib = _load()
    b = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.oracle_e2m1_to_f64(int(v)) for v in b], dtype=np.float64)


def e4m3_to_f64(codes) -> np.ndarray:
    lib = _load()
    b = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.oracle_e4m3_to_f64(int(v)) for v in b], dtype=np.float64)


def _x_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16 or x.ndim != 2:
        raise TypeError("x must be a 2-D float16 (or uint16 bit) array [M][K]")
    return x


def _cols(cols, N):
    if cols is None:
        return None, N
    c = np.ascontiguousarray(np.asarray(cols, dtype=np.int64).ravel())
    if c.size and (c.min() < 0 or c.max() >= N):
        raise IndexError("column index out of range")
    return c, int(c.size)


def nvfp4_linear(x, codes, scales, gscale, cols=None):
    """Reference NVFP4 linear.  Returns (y, l1), both float64 [M][ncols].

    x: float16 [M][K]; codes: uint8 [N][K/2] (low nibble = even k);
    scales: uint8 [N][K/16] (E4M3); gscale: FP32 tensor scale;
    cols: optional output columns to compute (default: all N).
    """
    xb = _x_bits(x)
    M, K = xb.shape
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    N = codes.shape[0]
    if K % 16 or codes.shape != (N, K // 2) or scales.shape != (N, K // 16):
        raise ValueError("bad NVFP4 shapes")
    c, nc = _cols(cols, N)
    y = np.zeros((M, nc), np.float64)
    l1 = np.zeros((M, nc), np.float64)
    _load().oracle_nvfp4_linear(M, N, K, _ptr(xb), _ptr(codes), _ptr(scales),
                                float(np.float32(gscale)),
                                None if c is None else _ptr(c), nc, _ptr(y), _ptr(l1))
    return y, l1


def fp8_linear(x, codes, scales, cols=None):
    """Reference FP8 (E4M3, 128x128 FP32 block scales) linear -> (y, l1) float64.

    codes: uint8 [N][K]; scales: float32 [ceil(N/128)][ceil(K/128)].
    """
    xb = _x_bits(x)
    M, K = xb.shape
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    N = codes.shape[0]
    if codes.shape != (N, K) or scales.shape != ((N + 127) // 128, (K + 127) // 128):
        raise ValueError("bad FP8 shapes")
    c, nc = _cols(cols, N)
    y = np.zeros((M, nc), np.float64)
    l1 = np.zeros((M, nc), np.float64)
    _load().oracle_fp8_linear(M, N, K, _ptr(xb), _ptr(codes), _ptr(scales),
                              None if c is None else _ptr(c), nc, _ptr(y), _ptr(l1))
    return y, l1


def argmax_rows(y) -> np.ndarray:
    """Lowest index of the row maximum (NaN skipped) for a float64 [M][N] array."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    M, N = y.shape
    idx = np.zeros(M, np.int64)
    _load().oracle_argmax_rows(M, N, _ptr(y), _ptr(idx))
    return idx


def verify(target, draft) -> tuple:
    """Greedy verification of a speculative round (oracle.c oracle_verify):
    (accepted drafts a, bonus token target[a])."""
    target = np.ascontiguousarray(target, dtype=np.int64)
    M = target.shape[0]
    draft = np.ascontiguousarray(np.asarray(draft, dtype=np.int32).reshape(-1)[:max(M - 1, 0)])
    if draft.shape[0] < M - 1:
        raise ValueError("need M - 1 draft tokens")
    out = np.zeros(2, np.int64)
    _load().oracle_verify(M, _ptr(target), _ptr(draft) if draft.size else None, _ptr(out))
    return int(out[0]), int(out[1])


def tolerance(l1, f16_out: bool = False, y_ref=None):
    """Accuracy contract: 1e-3 * sum|x*w| + 1e-6, plus one FP16 ulp of y_ref for
    FP16 output (ulp16(v) = 2^(max(floor(log2|v|), -14) - 10))."""
    tol = 1e-3 * np.asarray(l1, np.float64) + 1e-6
    if f16_out:
        a = np.abs(np.asarray(y_ref, np.float64))
        with np.errstate(divide="ignore"):
            e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
        e = np.maximum(np.where(a > 0, e, -14.0), -14.0)
        tol = tol + np.exp2(e - 10.0)
    return tol
