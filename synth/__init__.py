"""Seeded synthetic inputs for the skinny weight-only linear layer.

This module is shared by the tests, the smoke check and the benchmark: it
produces the inputs that both the CUDA path and the CPU oracle consume.  It
holds none of the method's arithmetic (no decoding, no products, no sums); the
one piece of number-format work here, rounding FP8 weights to E4M3 when they
are generated, is delegated to PyTorch's ``float8_e4m3fn`` conversion.

Recipes (one per weight format, matching the workloads the library targets):

* x: FP16, each element N(0, 1) drawn in float64 and rounded to FP16.
* NVFP4 weights: every E2M1 nibble uniform on 0..15 (so every code byte is
  uniform on 0..255, negative zero included); every E4M3 block scale uniform
  over the 65 positive codes 0x18..0x58, i.e. 2^-4 .. 2^4 (uniform in code,
  not in value); FP32 tensor scale float32(0.01).
* FP8 weights: w ~ N(0, 0.02) in float32; per 128x128 block (ragged blocks at
  the edges included) scale = absmax / 448 in float32 (1.0 for an all-zero
  block); code = E4M3 round-to-nearest-even of clamp(w / scale, -448, 448).

Every tensor comes from its own numpy PCG64 stream keyed by
(seed, tensor kind, shape...), so inputs do not depend on generation order.
"""
from __future__ import annotations

import numpy as np

NVFP4_GSCALE = np.float32(0.01)
SCALE_CODE_LO, SCALE_CODE_HI = 0x18, 0x58       # E4M3 2^-4 .. 2^4
_KIND = {"x": 1, "nvfp4": 2, "fp8": 3}


def rng(seed: int, kind: str, *ids: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(
        [int(seed), _KIND[kind], *[int(i) for i in ids]])))


def x_f16(M: int, K: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """Activations, float16 [M][K], N(0,1) rounded to FP16."""
    g = rng(seed, "x", M, K, stream)
    return g.standard_normal((M, K)).astype(np.float16)


def nvfp4_weights(N: int, K: int, seed: int = 0, stream: int = 0):
    """(codes u8[N][K/2], scales u8[N][K/16], gscale float32)."""
    if K % 16:
        raise ValueError("NVFP4 needs K % 16 == 0")
    g = rng(seed, "nvfp4", N, K, stream)
    codes = np.frombuffer(g.bytes(N * (K // 2)), dtype=np.uint8).reshape(N, K // 2).copy()
    scales = (g.integers(0, SCALE_CODE_HI - SCALE_CODE_LO + 1, size=(N, K // 16),
                         dtype=np.uint8) + np.uint8(SCALE_CODE_LO)).astype(np.uint8)
    return codes, scales, NVFP4_GSCALE


def fp8_quantize(w: np.ndarray):
    """float32 [N][K] -> (codes u8[N][K], scales f32[ceil(N/128)][ceil(K/128)])."""
    import torch

    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    nb, kb = (N + 127) // 128, (K + 127) // 128
    if N % 128 or K % 128:
        pad = np.zeros((nb * 128, kb * 128), np.float32)
        pad[:N, :K] = w
    else:
        pad = w
    blocks = pad.reshape(nb, 128, kb, 128)
    amax = np.abs(blocks).max(axis=(1, 3)).astype(np.float32)
    scales = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = blocks / scales[:, None, :, None]
    np.clip(q, np.float32(-448.0), np.float32(448.0), out=q)
    q = np.ascontiguousarray(q.reshape(nb * 128, kb * 128)[:N, :K])
    codes = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return np.ascontiguousarray(codes), scales


def fp8_weights(N: int, K: int, seed: int = 0, stream: int = 0):
    """(codes u8[N][K], scales f32[ceil(N/128)][ceil(K/128)]) from N(0, 0.02)."""
    g = rng(seed, "fp8", N, K, stream)
    w = g.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(0.02)
    return fp8_quantize(w)


# The decoder-layer shapes (K, N) of the 27B model the pages serve, unsharded.
LAYER_SHAPES = {
    "qkv": (5120, 7168),
    "o_proj": (6144, 5120),
    "gate_up": (5120, 34816),
    "down": (17408, 5120),
}
LM_HEAD_SHAPE = (5120, 151936)
