"""Concurrent streams with workspaces of their own (sk_stream_workspace).

Two streams each get a workspace; split-K calls of two different layers are
submitted to them alternately with no synchronisation in between, so their
kernels overlap on the GPU.  Every result must equal the stream's result when
it ran alone, bitwise (each stream's sums keep their fixed order), and match
the oracle; neither stream may report a bounded wait that ran out (the
cooperative launch keeps each persistent grid whole)."""
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
    yield skm
    assert skm.last_device_error() == skm.SK_OK


def test_two_streams_overlap(sk):
    import torch

    M = 8
    Ka, Na = 5120, 8704                       # NVFP4, five k-chunks (split-K)
    Kb, Nb = 6144, 5120                       # FP8, six k-chunks
    xa, xb = synth.x_f16(M, Ka, seed=31), synth.x_f16(M, Kb, seed=32)
    ca, sa, ga = synth.nvfp4_weights(Na, Ka, seed=33)
    cb, sb = synth.fp8_weights(Nb, Kb, seed=34)
    da = (dev(xa), dev(ca), dev(sa))
    db = (dev(xb), dev(cb), dev(sb))
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    sk.stream_workspace(s1)
    sk.stream_workspace(s2)
    try:
        ref_a = sk.nvfp4_gemm(*da, float(ga), stream=s1)
        ref_b = sk.fp8_gemm(*db, stream=s2)
        torch.cuda.synchronize()
        ref_a, ref_b = host(ref_a), host(ref_b)
        ya = [torch.full((M, Na), float("nan"), device="cuda:0") for _ in range(12)]
        yb = [torch.full((M, Nb), float("nan"), device="cuda:0") for _ in range(12)]
        torch.cuda.synchronize()
        for r in range(12):
            sk.nvfp4_gemm(*da, float(ga), y=ya[r], stream=s1)
            sk.fp8_gemm(*db, y=yb[r], stream=s2)
        assert sk.last_device_error(s1) == sk.SK_OK
        assert sk.last_device_error(s2) == sk.SK_OK
        for r in range(12):
            assert np.array_equal(host(ya[r]), ref_a), r
            assert np.array_equal(host(yb[r]), ref_b), r
        y_ref, l1 = oracle.nvfp4_linear(xa, ca, sa, ga)
        check(ref_a, y_ref, l1, False, "stream 1 nvfp4")
        y_ref, l1 = oracle.fp8_linear(xb, cb, sb)
        check(ref_b, y_ref, l1, False, "stream 2 fp8")
    finally:
        sk.stream_workspace(s1, 0)
        sk.stream_workspace(s2, 0)


def test_stream_workspace_serves_lm_head_and_quantizer(sk):
    import torch

    M, K, N = 4, 2048, 3001
    x = synth.x_f16(M, K, seed=41)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=42)
    w = (np.random.default_rng(43).standard_normal((512, 1024)) * 0.02).astype(np.float16)
    s = torch.cuda.Stream()
    sk.stream_workspace(s, 8 << 20)
    try:
        logits, am = sk.lm_head_argmax(dev(x), dev(codes), dev(scales), float(g), stream=s)
        c4, s4, g4 = sk.nvfp4_quantize(dev(w), stream=s)
        assert sk.last_device_error(s) == sk.SK_OK
        y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
        lg = host(logits)
        check(lg, y_ref, l1, False, "lm_head on a stream workspace")
        assert all(int(host(am)[m]) == int(np.argmax(lg[m])) for m in range(M))
        rc, rs, rg = oracle.quantize_nvfp4(w)
        assert np.array_equal(host(c4), rc) and np.array_equal(host(s4), rs)
        assert np.float32(host(g4)[0]) == np.float32(rg)
    finally:
        sk.stream_workspace(s, 0)


_FRESH = r"""
import sys
sys.path.insert(0, {root!r})
import numpy as np, torch
torch.cuda.set_device(0)
import fp8_weight_only_skinny_gb300 as sk     # no sk_init() in this process
import oracle, synth
M, K, N = 8, 3072, 700
x = synth.x_f16(M, K, seed=51)
codes, scales, g = synth.nvfp4_weights(N, K, seed=52)
xd, cd, sd = (torch.from_numpy(a).to("cuda:0") for a in (x, codes, scales))
s, other = torch.cuda.Stream(), torch.cuda.Stream()
try:
    sk.nvfp4_gemm(xd, cd, sd, float(g), stream=other)
    raise SystemExit("expected SK_ERR_NOT_INITIALIZED")
except sk.SkinnyError as e:
    assert e.status == sk.SK_ERR_NOT_INITIALIZED
sk.stream_workspace(s, 16 << 20)
y = sk.nvfp4_gemm(xd, cd, sd, float(g), stream=s)
s.synchronize()
y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - y_ref) <= oracle.tolerance(l1))
assert sk.last_device_error(s) == 0
print("fresh stream workspace ok")
"""


def test_stream_workspace_needs_no_sk_init():
    r = subprocess.run([sys.executable, "-c", _FRESH.format(root=ROOT)], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "fresh stream workspace ok" in r.stdout
