"""GPU parity at a very large N: 2^22 rows = 2^18 row groups of 16, with two
k-chunks so that every row group goes through the split-K fix-up (2^19 units
of partial sums at M = 1); and the same shape reported, not run, where its
partial sums exceed the workspace."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import check, dev, host

pytestmark = pytest.mark.gpu

N_MAX, K = 1 << 22, 2048


@pytest.fixture(scope="module")
def sk():
    import torch

    torch.cuda.set_device(0)
    import fp8_weight_only_skinny_gb300 as skm

    skm.init()
    yield skm
    assert skm.last_device_error() == skm.SK_OK


def _edge_rows(n_random, seed):
    fixed = [0, 1, 15, 16, N_MAX // 2, N_MAX - 17, N_MAX - 16, N_MAX - 1]
    return np.unique(np.concatenate([fixed, np.random.default_rng(seed).choice(N_MAX, n_random, replace=False)]))


def test_nvfp4_at_four_million_rows(sk):
    import torch

    g = torch.Generator(device="cuda:0")
    g.manual_seed(5)
    codes = torch.randint(0, 256, (N_MAX, K // 2), dtype=torch.uint8, device="cuda:0", generator=g)
    scales = torch.randint(0x18, 0x59, (N_MAX, K // 16), dtype=torch.uint8, device="cuda:0", generator=g)
    x = synth.x_f16(1, K, seed=77)
    y = host(sk.nvfp4_gemm(dev(x), codes, scales, 0.01))
    rows = _edge_rows(120, 1)
    ri = torch.from_numpy(rows).to("cuda:0")
    y_ref, l1 = oracle.nvfp4_linear(x, host(codes[ri]), host(scales[ri]), np.float32(0.01))
    check(y[:, rows], y_ref, l1, False, "nvfp4 N = 2^22")
    # two tokens take the tensor-core variant, whose partials (2^19 units x 512 B) exceed the
    # default workspace: reported before any launch
    with pytest.raises(sk.SkinnyError) as e:
        sk.nvfp4_gemm(dev(synth.x_f16(2, K, seed=78)), codes, scales, 0.01)
    assert sk.STATUS[e.value.status] == "SK_ERR_WORKSPACE"
    del codes, scales
    torch.cuda.empty_cache()


def test_fp8_at_four_million_rows(sk):
    import torch

    g = torch.Generator(device="cuda:0")
    g.manual_seed(6)
    codes = torch.randint(0, 0x7F, (N_MAX, K), dtype=torch.uint8, device="cuda:0", generator=g)   # no NaN codes
    codes |= torch.randint(0, 2, (N_MAX, K), dtype=torch.uint8, device="cuda:0", generator=g) << 7
    scales = torch.rand((N_MAX // 128, K // 128), device="cuda:0", generator=g) * 0.02 + 0.001
    x = synth.x_f16(1, K, seed=79)
    y = host(sk.fp8_gemm(dev(x), codes, scales))
    blocks = np.unique(np.concatenate([[0, 1, N_MAX // 256, N_MAX // 128 - 1],
                                       np.random.default_rng(2).choice(N_MAX // 128, 4, replace=False)]))
    rows = np.concatenate([np.arange(b * 128, (b + 1) * 128) for b in blocks])
    ri, bi = torch.from_numpy(rows).to("cuda:0"), torch.from_numpy(blocks).to("cuda:0")
    y_ref, l1 = oracle.fp8_linear(x, host(codes[ri]), host(scales[bi]))
    check(y[:, rows], y_ref, l1, False, "fp8 N = 2^22")
    del codes, scales
    torch.cuda.empty_cache()
