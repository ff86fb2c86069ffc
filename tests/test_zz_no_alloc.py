"""nvfp4_gemm_noalloc: the NVFP4 linear for callers that cannot allocate
device memory (an arena or pool allocator that owns all device memory, an
allocator frozen after start-up, a serving path with a no-allocation rule).

It runs the same kernel as nvfp4_gemm but keeps its split-K scratch in a
static device array instead of the sk_init() workspace.  The test calls it
through the C ABI twice in a row (the array keeps the first call's contents)
and checks each result against nvfp4_gemm on the same inputs, within the
accuracy contract and bitwise (same kernel, same grid, same sum order).  This
file runs last so that a failure here leaves every other test already run.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import check, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    import torch

    torch.cuda.set_device(0)
    import fp8_weight_only_skinny_gb300 as skm

    skm.init()
    return skm


@pytest.mark.parametrize("M,K,N", [(1, 2048, 1000), (8, 3072, 500), (4, 512, 64), (8, 1024, 40)])
def test_noalloc_matches_nvfp4_gemm_on_two_calls(sk, M, K, N):
    import torch

    x = synth.x_f16(M, K, seed=M + K)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=N + 3)
    xd, cd, sd = dev(x), dev(codes), dev(scales)
    ref = host(sk.nvfp4_gemm(xd, cd, sd, float(g)))
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    tol = oracle.tolerance(l1)
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda:0")
        st = sk.lib.nvfp4_gemm_noalloc(xd.data_ptr(), cd.data_ptr(), sd.data_ptr(), float(g), y.data_ptr(),
                                       M, N, K, None)
        assert st == sk.SK_OK, sk.status_string(st)
        yh = host(y)
        assert np.all(np.abs(yh - ref) <= tol)
        assert np.array_equal(yh, ref)
        check(yh, y_ref, l1, False, "noalloc vs oracle")


def test_noalloc_rejects_shapes_beyond_its_scratch(sk):
    import torch

    # M=8, K=5120 (5 chunks): 2867 row groups fit in ~7 MiB of partials; 4096 do not.
    x = torch.zeros((8, 5120), dtype=torch.float16, device="cuda:0")
    codes = torch.zeros((65536, 2560), dtype=torch.uint8, device="cuda:0")
    scales = torch.zeros((65536, 320), dtype=torch.uint8, device="cuda:0")
    y = torch.zeros((8, 65536), dtype=torch.float32, device="cuda:0")
    st = sk.lib.nvfp4_gemm_noalloc(x.data_ptr(), codes.data_ptr(), scales.data_ptr(), 1.0, y.data_ptr(),
                                   8, 65536, 5120, None)
    assert st == 7, sk.status_string(st)         # SK_ERR_WORKSPACE, nothing launched
    assert sk.lib.nvfp4_gemm_noalloc(x.data_ptr(), codes.data_ptr(), scales.data_ptr(), 1.0, y.data_ptr(),
                                     9, 16, 5120, None) == 1
