"""GPU parity with the grid capped to a few CTAs, so every CTA walks many
units: the TMA ring wraps around many times, both consumer groups alternate
over ring stages, the activations are reloaded at k-chunk changes, and the
split-K fix-up runs with several units and row groups per CTA."""
import os

import numpy as np
import pytest

import oracle
import synth
from gpu_util import Guarded, argmax_ok, check, dev, host, variant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    import torch

    torch.cuda.set_device(0)
    import fp8_weight_only_skinny_gb300 as skm

    skm.init()
    yield skm
    assert skm.last_device_error() == skm.SK_OK


@pytest.fixture(params=[1, 3, 7])
def max_ctas(request):
    os.environ["SK_MAX_CTAS"] = str(request.param)
    yield request.param
    del os.environ["SK_MAX_CTAS"]


MV = [(1, "simt"), (1, "tensor"), (2, "auto"), (4, "auto"), (8, "auto")]


@pytest.mark.parametrize("M,var", MV)
# K = 10240: ten k-chunks, the owners' many-chunk sums, each owner summing
# several row groups in turn on the capped grids.
@pytest.mark.parametrize("K,N", [(1024, 520), (3072, 200), (5120, 96), (10240, 520)])
def test_nvfp4_many_units_per_cta(sk, max_ctas, M, var, K, N):
    x = synth.x_f16(M, K, seed=K + M)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=N + 1)
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    import torch

    out = Guarded((M, N), torch.float32)
    with variant(sk, var):
        sk.nvfp4_gemm(dev(x), dev(codes), dev(scales), float(g), y=out.t)
    check(out.host("nvfp4 output"), y_ref, l1, False, f"nvfp4 ctas={max_ctas} M{M} K{K} N{N}")


@pytest.mark.parametrize("M,var", MV)
@pytest.mark.parametrize("K,N", [(1024, 520), (3072, 200), (4096, 130), (10240, 264)])
def test_fp8_many_units_per_cta(sk, max_ctas, M, var, K, N):
    x = synth.x_f16(M, K, seed=K + M + 5)
    codes, scales = synth.fp8_weights(N, K, seed=N + 2)
    y_ref, l1 = oracle.fp8_linear(x, codes, scales)
    import torch

    out = Guarded((M, N), torch.float16)
    with variant(sk, var):
        sk.fp8_gemm(dev(x), dev(codes), dev(scales), y=out.t, f16_out=True)
    check(out.host("fp8 output"), y_ref, l1, True, f"fp8 ctas={max_ctas} M{M} K{K} N{N}")


@pytest.mark.parametrize("M,var", [(1, "simt"), (1, "tensor"), (8, "auto")])
def test_lm_head_many_units_per_cta(sk, max_ctas, M, var):
    K, N = 2048, 1000
    x = synth.x_f16(M, K, seed=77 + M)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=78)
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    import torch

    glg, gam = Guarded((M, N), torch.float32), Guarded((M,), torch.int32, fill=-7)
    with variant(sk, var):
        sk.lm_head_argmax(dev(x), dev(codes), dev(scales), float(g), logits=glg.t, argmax=gam.t)
    lg, am = glg.host("logits"), gam.host("argmax")
    check(lg, y_ref, l1, False, "lm_head few CTAs")
    argmax_ok(am, y_ref, l1, lg)


def test_results_do_not_depend_on_grid(sk):
    """Each grid size fixes its own summation order: repeated calls on one grid
    are bitwise identical and every grid meets the accuracy contract."""
    M, K, N = 8, 3072, 300
    x = synth.x_f16(M, K, seed=3)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=3)
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    outs = []
    for cap in ("2", "5", "1000"):
        os.environ["SK_MAX_CTAS"] = cap
        try:
            a = host(sk.nvfp4_gemm(dev(x), dev(codes), dev(scales), float(g)))
            b = host(sk.nvfp4_gemm(dev(x), dev(codes), dev(scales), float(g)))
        finally:
            del os.environ["SK_MAX_CTAS"]
        assert np.array_equal(a, b)
        check(a, y_ref, l1, False, f"grid cap {cap}")
        outs.append(a)
