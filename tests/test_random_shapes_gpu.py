"""GPU parity on seeded random shapes: both formats, M = 1..8, ragged N (any
residue modulo the 16-row group and the 128-row FP8 scale block), K over one
to several k-chunks with ragged last chunks, each kernel variant, FP32 and
FP16 output, activations 32-byte aligned or only 16 -- every output element
against the oracle, every output between guard bands.  The cases are drawn
from one fixed seed, so a failure names a reproducible shape."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import Guarded, check, dev, variant

pytestmark = pytest.mark.gpu

N_CASES = 96


def _cases():
    r = np.random.default_rng(20261203)
    out = []
    for i in range(N_CASES):
        fmt = "nvfp4" if i % 2 == 0 else "fp8"
        kq = 256 if fmt == "nvfp4" else 128          # the formats' K granularity
        K = int(kq * r.integers(1, 3 * 1024 // kq + 1))   # up to 3 k-chunks
        N = int(r.integers(1, 700))
        M = int(r.integers(1, 9))
        var = ("auto", "tensor", "simt")[int(r.integers(0, 3))] if M == 1 else "auto"
        f16 = bool(r.integers(0, 2))
        off = int(r.integers(0, 2)) * 8              # halves: x 32-byte aligned or 16 bytes past
        out.append((fmt, M, N, K, var, f16, off, 1000 + i))
    return out


@pytest.fixture(scope="module")
def sk():
    import torch

    torch.cuda.set_device(0)
    import fp8_weight_only_skinny_gb300 as skm

    skm.init()
    yield skm
    assert skm.last_device_error() == skm.SK_OK


@pytest.mark.parametrize("fmt,M,N,K,var,f16,off,seed", _cases())
def test_random_shape(sk, fmt, M, N, K, var, f16, off, seed):
    import torch

    x = synth.x_f16(M, K, seed=seed)
    buf = torch.zeros(M * K + 16, dtype=torch.float16, device="cuda:0")
    xd = buf[off:off + M * K].view(M, K)
    xd.copy_(dev(x))
    y = Guarded((M, N), torch.float16 if f16 else torch.float32)
    with variant(sk, var):
        if fmt == "nvfp4":
            codes, scales, g = synth.nvfp4_weights(N, K, seed=seed + 1)
            sk.nvfp4_gemm(xd, dev(codes), dev(scales), float(g), y=y.t, f16_out=f16)
            y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
        else:
            codes, scales = synth.fp8_weights(N, K, seed=seed + 1)
            sk.fp8_gemm(xd, dev(codes), dev(scales), y=y.t, f16_out=f16)
            y_ref, l1 = oracle.fp8_linear(x, codes, scales)
    check(y.host(f"{fmt} output"), y_ref, l1, f16, f"{fmt} M{M} N{N} K{K} {var} f16={f16} off={off}")
