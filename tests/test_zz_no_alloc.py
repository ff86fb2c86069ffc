"""nvfp4_gemm_noalloc: the NVFP4 linear for callers that cannot allocate
device memory (an arena or pool allocator that owns all device memory, an
allocator frozen after start-up, a serving path with a no-allocation rule).

It runs the same kernel as nvfp4_gemm but keeps its split-K scratch in a
static device array instead of the sk_init() workspace.  The tests call it
through the C ABI twice in a row (the array keeps the first call's contents)
and check each result against nvfp4_gemm on the same inputs, within the
accuracy contract and bitwise (same kernel, same grid, same sum order); check
the scratch limit on both sides of the boundary; run a first call in a fresh
process that never calls sk_init(); and check that a call whose bounded waits
ran out is followed by a correct one.  This file runs last so that a failure
here leaves every other test already run.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import synth
from gpu_util import check, dev, host

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sk():
    import torch

    torch.cuda.set_device(0)
    import fp8_weight_only_skinny_gb300 as skm

    skm.init()
    return skm


def _noalloc(sk, xd, cd, sd, g, y, M, N, K):
    return sk.lib.nvfp4_gemm_noalloc(xd.data_ptr(), cd.data_ptr(), sd.data_ptr(), float(g), y.data_ptr(),
                                     M, N, K, None)


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
        st = _noalloc(sk, xd, cd, sd, g, y, M, N, K)
        assert st == sk.SK_OK, sk.status_string(st)
        yh = host(y)
        assert np.all(np.abs(yh - ref) <= tol)
        assert np.array_equal(yh, ref)
        check(yh, y_ref, l1, False, "noalloc vs oracle")


@pytest.mark.parametrize("M", [2, 8])
def test_noalloc_scratch_limit_boundary(sk, M):
    """At K = 5120 (five 1024-k chunks) every M >= 2 uses 8 token slots, so the
    partial sums take ceil(N/16) * 5 * 512 bytes of the 8,384,512 available:
    N = 52,400 fits and N = 52,416 (one more row group) is rejected with
    SK_ERR_WORKSPACE before anything is launched."""
    import torch

    K, N_in, N_out = 5120, 52400, 52416
    x = torch.zeros((M, K), dtype=torch.float16, device="cuda:0")
    codes = torch.zeros((N_out, K // 2), dtype=torch.uint8, device="cuda:0")
    scales = torch.full((N_out, K // 16), 0x38, dtype=torch.uint8, device="cuda:0")
    y = torch.full((M, N_out), float("nan"), dtype=torch.float32, device="cuda:0")
    assert _noalloc(sk, x, codes, scales, 1.0, y, M, N_out, K) == sk.SK_ERR_WORKSPACE
    assert torch.isnan(y).all().item()                      # nothing ran
    st = _noalloc(sk, x, codes, scales, 1.0, y, M, N_in, K)
    assert st == sk.SK_OK, sk.status_string(st)
    flat = host(y.view(-1))                                   # y is [M][N_in] row-major at this N
    assert (flat[:M * N_in] == 0).all()
    assert np.isnan(flat[M * N_in:]).all()
    assert sk.lib.nvfp4_gemm_noalloc(x.data_ptr(), codes.data_ptr(), scales.data_ptr(), 1.0, y.data_ptr(),
                                     9, 16, K, None) == sk.SK_ERR_INVALID_ARG


_FRESH = r"""
import sys
sys.path.insert(0, {root!r})
import numpy as np, torch
torch.cuda.set_device(0)
import fp8_weight_only_skinny_gb300 as sk   # loads the library; no sk_init() anywhere below
import oracle, synth
M, K, N = 8, 5120, 700                       # five k-chunks: the split-K path
x = synth.x_f16(M, K, seed=41)
codes, scales, g = synth.nvfp4_weights(N, K, seed=42)
xd, cd, sd = (torch.from_numpy(a).to("cuda:0") for a in (x, codes, scales))
outs = []
for _ in range(2):
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda:0")
    st = sk.lib.nvfp4_gemm_noalloc(xd.data_ptr(), cd.data_ptr(), sd.data_ptr(), float(g), y.data_ptr(),
                                   M, N, K, None)
    assert st == 0, st
    torch.cuda.synchronize()
    outs.append(y.cpu().numpy().astype(np.float64))
y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
assert np.all(np.abs(outs[0] - y_ref) <= oracle.tolerance(l1)), "first call outside the tolerance"
assert np.array_equal(outs[0], outs[1]), "second call differs from the first"
print("fresh-process noalloc ok")
"""


def test_noalloc_first_call_in_a_fresh_process_without_sk_init():
    """The first call on a device does its own set-up (symbol address, tensor
    map encoder, SM count): in a process that never calls sk_init(), a split-K
    shape matches the oracle and a second call matches the first bitwise."""
    r = subprocess.run([sys.executable, "-c", _FRESH.format(root=ROOT)], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "fresh-process noalloc ok" in r.stdout


def test_noalloc_recovers_after_a_timed_out_call(sk):
    """With the failure-injection hook the kernel issues no weight copies, its
    bounded waits run out (about one second) and it leaves garbage and counts
    in the static scratch.  The next call clears what must start at zero, so it
    matches nvfp4_gemm bitwise again."""
    import torch

    M, K, N = 8, 3072, 500
    x = synth.x_f16(M, K, seed=51)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=52)
    xd, cd, sd = dev(x), dev(codes), dev(scales)
    ref = host(sk.nvfp4_gemm(xd, cd, sd, float(g)))
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda:0")
    sk.lib.sk_inject_wait_timeout(1)
    assert _noalloc(sk, xd, cd, sd, g, y, M, N, K) == sk.SK_OK
    torch.cuda.synchronize()
    for _ in range(2):
        y.fill_(float("nan"))
        assert _noalloc(sk, xd, cd, sd, g, y, M, N, K) == sk.SK_OK
        assert np.array_equal(host(y), ref)
    assert sk.last_device_error() == sk.SK_OK           # the sk_init workspace saw no timeout
