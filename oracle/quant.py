"""CPU oracle for the weight quantizers (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU leg may
import this module; the CUDA path shares nothing with it.

What is computed.  The pages convert an FP16/BF16 checkpoint to NVFP4 (block-
wise 4-bit floating point: v100-skinny ai-manual.ru article, section
"Конвертация модели в NVFP4"; page "NVFP4 在 Volta 上！", v1.1 section: FP4
regions stay FP4, FP8 regions stay FP8) but print no rounding rules.  This
library fixes the plainest reading, with every step an IEEE binary32
operation rounded to nearest-even, in this order:

  FP8-E4M3 with one FP32 scale per 128 x 128 block:
    a = max |w| over the block;  s = a / 448  (s = 1 when a = 0)
    code = E4M3(w / s), round to nearest, ties to even, saturating at +-448

  NVFP4 (two-level scale):
    A = max |w| over the tensor;  G = A / 2688  (2688 = 448 * 6; G = 1 when A = 0)
    per row and 16 consecutive k:  b = max |w| over the 16
      t = (b / 6) / G;  sc = E4M3(t)  (nearest-even, saturating);  S = value(sc)
      code = E2M1(w / (S * G)), nearest-even, saturating at +-6
      (S = 0: every code is a signed zero)

Rounding to E4M3 / E2M1 is done by brute force against the format's table of
values (decoded from the bit fields by oracle.e4m3_to_f64 / e2m1_to_f64):
the nearest value wins, a tie goes to the code with an even mantissa (bit 0
clear), and the sign of the input (including -0.0) is kept.

Parity status: pinned (tests/test_oracle_quant.py).
"""
from __future__ import annotations

import numpy as np

from .oracle import e2m1_to_f64, e4m3_to_f64

_F32 = np.float32


def _table(decode, codes):
    vals = decode(np.array(codes))
    order = np.argsort(vals, kind="stable")
    return vals[order], np.array(codes)[order]


_E4M3_POS = _table(e4m3_to_f64, [c for c in range(0x7F)])          # 0x00..0x7E (0x7F is NaN)
_E2M1_POS = _table(e2m1_to_f64, list(range(8)))                     # 0, 0.5, ..., 6


def _round_to_table(v, table, sign_bit):
    """Nearest-even rounding of float32 values v onto a sign-magnitude format
    whose positive values and codes are `table`; saturates at its maximum."""
    vals, codes = table
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), vals[-1])
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((codes[hi] & 1) == 0) & ((codes[lo] & 1) == 1))
    out = np.where(pick_hi, codes[hi], codes[lo]).astype(np.int64)
    out = np.where(a == vals[lo], codes[lo], out)
    return np.where(np.signbit(v), out | sign_bit, out).astype(np.uint8)


def e4m3_round(v):
    """float32 values -> E4M3 codes (nearest-even, saturating, sign kept)."""
    return _round_to_table(np.asarray(v, dtype=_F32), _E4M3_POS, 0x80)


def e2m1_round(v):
    """float32 values -> E2M1 codes 0..15 (nearest-even, saturating, sign kept)."""
    return _round_to_table(np.asarray(v, dtype=_F32), _E2M1_POS, 0x8)


def quantize_fp8(w):
    """FP16 [N][K] -> (codes u8 [N][K], scales f32 [ceil(N/128)][ceil(K/128)])."""
    w = np.asarray(w, dtype=np.float16).astype(_F32)
    N, K = w.shape
    nb, kb = (N + 127) // 128, (K + 127) // 128
    codes = np.zeros((N, K), np.uint8)
    scales = np.ones((nb, kb), _F32)
    for i in range(nb):
        for j in range(kb):
            blk = w[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            a = _F32(np.max(np.abs(blk)))
            s = _F32(a / _F32(448.0)) if a > 0 else _F32(1.0)
            scales[i, j] = s
            codes[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128] = e4m3_round((blk / s).astype(_F32))
    return codes, scales


def quantize_nvfp4(w, amax=None):
    """FP16 [N][K] (K % 16 == 0) -> (codes u8 [N][K/2], low nibble = even k;
    scales u8 [N][K/16]; tensor scale float32).

    amax: max |w| over the whole tensor when w holds only some of its rows
    (default: taken from w itself)."""
    w = np.asarray(w, dtype=np.float16).astype(_F32)
    N, K = w.shape
    if amax is not None:
        A = _F32(amax)
    else:
        A = _F32(np.max(np.abs(w))) if w.size else _F32(0.0)
    G = _F32(A / _F32(2688.0)) if A > 0 else _F32(1.0)
    blocks = w.reshape(N, K // 16, 16)
    b = np.max(np.abs(blocks), axis=2).astype(_F32)
    t = ((b / _F32(6.0)).astype(_F32) / G).astype(_F32)
    sc = e4m3_round(t)
    S = e4m3_to_f64(np.arange(256)).astype(_F32)[sc]
    denom = (S * G).astype(_F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (blocks / denom[:, :, None]).astype(_F32)
    nib = e2m1_round(q)
    zero = (S == 0)[:, :, None]
    nib = np.where(zero, np.where(np.signbit(blocks), 0x8, 0x0), nib).astype(np.uint8).reshape(N, K)
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return codes, sc.astype(np.uint8), G
