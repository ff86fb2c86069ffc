"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function that include/skinny.h declares,
and reject bad arguments with the documented status before touching the GPU.
Fake device pointers are only ever passed in combinations that a check ahead
of any CUDA call rejects (a misaligned pointer, a bad shape), so nothing here
can reach a launch.
"""
import ctypes
import os
import re

import pytest

import fp8_weight_only_skinny_gb300 as sk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "include", "skinny.h")

OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3


def _declared():
    txt = open(HDR).read()
    return re.findall(r"SK_API\s+[\w\s\*]+?\b(\w+)\s*\(", txt)


def test_library_exports_every_declared_symbol():
    names = _declared()
    assert len(names) >= 10
    lib = ctypes.CDLL(sk.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in skinny.h but not exported"
    assert set(names) == set(sk.EXPORTS)


def test_status_strings():
    for code, name in sk.STATUS.items():
        assert sk.status_string(code).startswith(name)
    assert "unknown" in sk.status_string(99)
    assert sk.lib.sk_version() >= 100


A = 0x10000          # a 16-byte-aligned fake device address (never dereferenced)


def _nv(x=A, c=A, s=A, y=A, M=1, N=16, K=256):
    return sk.lib.nvfp4_gemm(x, c, s, 1.0, y, M, N, K, None)


def _f8(x=A, c=A, s=A, y=A, M=1, N=16, K=128):
    return sk.lib.fp8_gemm(x, c, s, y, M, N, K, None)


def _lm(x=A, c=A, s=A, lg=A, am=A, M=1, N=16, K=256):
    return sk.lib.lm_head_argmax(x, c, s, 1.0, lg, am, M, N, K, None)


@pytest.mark.parametrize("M", [0, 9, -1])
def test_m_out_of_range(M):
    assert _nv(M=M) == INVALID
    assert _f8(M=M) == INVALID
    assert _lm(M=M) == INVALID


def test_negative_sizes_and_null_pointers():
    assert _nv(N=-1) == INVALID and _nv(K=-256) == INVALID
    assert _f8(N=-5) == INVALID
    assert _nv(x=None) == INVALID and _nv(c=None) == INVALID and _nv(s=None) == INVALID
    assert _nv(y=None) == INVALID
    assert _f8(s=None) == INVALID and _f8(y=None) == INVALID
    assert _lm(am=None) == INVALID
    assert _lm(N=0) == INVALID


@pytest.mark.parametrize("K", [16, 64, 128, 320, 1000])
def test_nvfp4_k_must_be_multiple_of_256(K):
    assert _nv(K=K) == UNSUPPORTED
    assert _lm(K=K) == UNSUPPORTED


@pytest.mark.parametrize("K", [16, 64, 100, 200])
def test_fp8_k_must_be_multiple_of_128(K):
    assert _f8(K=K) == UNSUPPORTED


def test_misaligned_pointers_rejected():
    assert _nv(x=A + 8) == MISALIGNED
    assert _nv(c=A + 4) == MISALIGNED
    assert _nv(s=A + 1) == MISALIGNED
    assert _nv(y=A + 2) == MISALIGNED
    assert sk.lib.nvfp4_gemm_f16out(A, A, A, 1.0, A + 1, 1, 16, 256, None) == MISALIGNED
    assert _f8(s=A + 2) == MISALIGNED
    assert _f8(c=A + 8) == MISALIGNED
    assert _lm(am=A + 2) == MISALIGNED
    assert _lm(lg=A + 2) == MISALIGNED


def test_variant_setting_round_trips_and_rejects_unknown_values():
    prev = sk.set_variant(sk.VARIANT_TENSOR)
    try:
        assert sk.set_variant(sk.VARIANT_SIMT) == sk.VARIANT_TENSOR
        assert sk.lib.sk_set_variant(3) == -1          # unknown: nothing changes
        assert sk.lib.sk_set_variant(-1) == -1
        with pytest.raises(ValueError):
            sk.set_variant(7)
        assert sk.set_variant(sk.VARIANT_AUTO) == sk.VARIANT_SIMT
    finally:
        sk.set_variant(prev)


def _vf(x=A, c=A, s=A, lg=A, am=A, dr=A, ac=A, M=2, N=16, K=256):
    return sk.lib.lm_head_verify(x, c, s, 1.0, lg, am, dr, ac, M, N, K, None)


def test_lm_head_verify_argument_checks():
    assert _vf(ac=None) == INVALID                 # accept is required
    assert _vf(dr=None) == INVALID                 # drafts are required when M > 1
    assert _vf(ac=A + 2) == MISALIGNED
    assert _vf(dr=A + 2) == MISALIGNED
    assert _vf(K=0) == UNSUPPORTED                 # nothing to verify against
    assert _vf(M=9) == INVALID


def test_quantizer_argument_checks():
    L = sk.lib
    assert L.fp8_quantize(A, A, A, -1, 128, None) == INVALID
    assert L.fp8_quantize(None, A, A, 4, 128, None) == INVALID
    assert L.fp8_quantize(A, A, A, 4, 12, None) == UNSUPPORTED        # K % 8
    assert L.fp8_quantize(A + 8, A, A, 4, 128, None) == MISALIGNED
    assert L.fp8_quantize(A, A, A, 0, 128, None) == OK               # empty: nothing to do
    assert L.nvfp4_quantize(A, A, A, None, 4, 256, None) == INVALID
    assert L.nvfp4_quantize(A, A, A, A, 4, 24, None) == UNSUPPORTED   # K % 16
    assert L.nvfp4_quantize(A, A + 4, A, A, 4, 256, None) == MISALIGNED


def _smp(lg=A, u=A, tok=A, T=0.6, k=10, p=0.9, M=2, N=4096, K=256):
    return sk.lib.lm_head_sample(A, A, A, 1.0, lg, u, T, k, p, tok, M, N, K, None)


def test_lm_head_sample_argument_checks():
    assert _smp(lg=None) == INVALID and _smp(u=None) == INVALID and _smp(tok=None) == INVALID
    assert _smp(k=0) == INVALID and _smp(k=4097) == INVALID       # 1 <= top_k <= N
    assert _smp(k=2000) == UNSUPPORTED                             # above 1024 candidates
    assert _smp(p=0.0) == INVALID and _smp(p=1.5) == INVALID and _smp(p=float("nan")) == INVALID
    assert _smp(u=A + 2) == MISALIGNED and _smp(tok=A + 2) == MISALIGNED
