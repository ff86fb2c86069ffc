"""Parity at the full decode-layer sizes, in the launch configuration the
benchmark uses (default grid, PDL on): every output column of every decode
shape against the oracle, the full-vocabulary lm_head with its fused argmax
checked against the oracle's own argmax over the whole row (with each kernel
variant at M = 1), and a CUDA-graph-replayed decode stack (the benchmark's
step structure, shortened)."""
import functools

import numpy as np
import pytest

import oracle
import synth
from gpu_util import Guarded, argmax_ok, check, dev, host, variant


@functools.lru_cache(maxsize=None)
def _nv(N, K, seed):
    return synth.nvfp4_weights(N, K, seed=seed)


@functools.lru_cache(maxsize=None)
def _f8(N, K, seed):
    return synth.fp8_weights(N, K, seed=seed)


@functools.lru_cache(maxsize=4)
def _head_ref(M):
    """Inputs and the oracle's logits over the whole vocabulary for the lm_head
    case at M rows (about 0.8 G exact products per row; computed once)."""
    K, N = synth.LM_HEAD_SHAPE
    x = synth.x_f16(M, K, seed=100 + M)
    codes, scales, g = _nv(N, K, 101)
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    return x, codes, scales, g, y_ref, l1

pytestmark = pytest.mark.gpu

SHAPES = [("qkv", 5120, 7168), ("o_proj", 6144, 5120), ("gate_up", 5120, 34816), ("down", 17408, 5120)]


@pytest.fixture(scope="module")
def sk():
    import torch

    torch.cuda.set_device(0)
    import fp8_weight_only_skinny_gb300 as skm

    skm.init()
    yield skm
    assert skm.last_device_error() == skm.SK_OK


def _cols(N, n=192, seed=0):
    r = np.random.default_rng(seed)
    # the first and last row groups, chunk-boundary rows and random ones
    fixed = [0, 1, 15, 16, N // 2, N - 17, N - 16, N - 1]
    return np.unique(np.concatenate([fixed, r.choice(N, n, replace=False)]))


@pytest.mark.parametrize("name,K,N", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_nvfp4_full_size(sk, name, K, N, M):
    """Every one of the N output columns against the oracle (FP32 output)."""
    import torch

    x = synth.x_f16(M, K, seed=K + M)
    codes, scales, g = _nv(N, K, N)
    y = Guarded((M, N), torch.float32)
    sk.nvfp4_gemm(dev(x), dev(codes), dev(scales), float(g), y=y.t)
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    check(y.host(f"nvfp4 {name}"), y_ref, l1, False, f"nvfp4 {name} M={M}")


@pytest.mark.parametrize("name,K,N", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_fp8_full_size(sk, name, K, N, M):
    """Every one of the N output columns against the oracle (FP16 output, as
    the benchmark's stack writes it)."""
    import torch

    x = synth.x_f16(M, K, seed=K + M + 1)
    codes, scales = _f8(N, K, N + 1)
    y = Guarded((M, N), torch.float16)
    sk.fp8_gemm(dev(x), dev(codes), dev(scales), y=y.t, f16_out=True)
    y_ref, l1 = oracle.fp8_linear(x, codes, scales)
    check(y.host(f"fp8 {name}"), y_ref, l1, True, f"fp8 {name} M={M}")


@pytest.mark.parametrize("M,var", [(1, "auto"), (1, "tensor"), (1, "simt"), (8, "auto")])
def test_lm_head_full_size(sk, M, var):
    """K=5120, N=151936: every logit against the oracle, and the fused pick
    against the oracle's lowest-index argmax of the whole row -- bit-exact
    wherever the oracle's top-2 gap exceeds the two tolerances -- as well as
    against the same call's FP32 logits, bitwise."""
    import torch

    x, codes, scales, g, y_ref, l1 = _head_ref(M)
    K, N = synth.LM_HEAD_SHAPE
    glg, gam = Guarded((M, N), torch.float32), Guarded((M,), torch.int32, fill=-7)
    with variant(sk, var):
        sk.lm_head_argmax(dev(x), dev(codes), dev(scales), float(g), logits=glg.t, argmax=gam.t)
        _, am_only = sk.lm_head_argmax(dev(x), dev(codes), dev(scales), float(g), want_logits=False)
    lg, am = glg.host("logits"), gam.host("argmax")
    check(lg, y_ref, l1, False, f"lm_head M={M} {var}")
    argmax_ok(am, y_ref, l1, lg)
    assert np.array_equal(host(am_only), am)


@pytest.mark.parametrize("M", [1, 8])
def test_graph_replayed_stack(sk, M):
    """Two decoder layers (qkv/o FP8, gate_up/down NVFP4) and the lm_head,
    captured once into a CUDA graph with PDL between the calls and replayed
    three times: every output equals the eager result bitwise and the oracle on
    sampled columns."""
    import torch

    layers = []
    for li in range(2):
        for name, K, N in SHAPES:
            fmt = "fp8" if name in ("qkv", "o_proj") else "nvfp4"
            x = synth.x_f16(M, K, seed=1000 * li + K)
            if fmt == "fp8":
                w = synth.fp8_weights(N, K, seed=2000 * li + N)
            else:
                w = synth.nvfp4_weights(N, K, seed=2000 * li + N)
            layers.append((name, fmt, x, w, tuple(dev(a) for a in (x, *w[:2])),
                           torch.empty((M, N), dtype=torch.float16, device="cuda:0")))
    K, N = synth.LM_HEAD_SHAPE
    hx = synth.x_f16(M, K, seed=7)
    hw = synth.nvfp4_weights(N, K, seed=8)
    hd = (dev(hx), dev(hw[0]), dev(hw[1]))
    logits = torch.empty((M, N), dtype=torch.float32, device="cuda:0")
    am = torch.empty((M,), dtype=torch.int32, device="cuda:0")

    def step():
        for name, fmt, x, w, d, y in layers:
            if fmt == "fp8":
                sk.fp8_gemm(d[0], d[1], d[2], y=y, f16_out=True)
            else:
                sk.nvfp4_gemm(d[0], d[1], d[2], float(w[2]), y=y, f16_out=True)
        sk.lm_head_argmax(hd[0], hd[1], hd[2], float(hw[2]), logits=logits, argmax=am)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step()
    s.synchronize()
    eager = [host(l[5]) for l in layers] + [host(logits), host(am)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    for _ in range(3):
        with torch.cuda.stream(s):                 # poison and replay on the same stream
            for l in layers:
                l[5].fill_(float("nan"))
            logits.fill_(float("nan"))
            g.replay()
        s.synchronize()
        got = [host(l[5]) for l in layers] + [host(logits), host(am)]
        for idx, (a, b) in enumerate(zip(got, eager)):
            assert np.array_equal(a, b), (idx, int(np.sum(~(a == b))), a.size)
    for (name, fmt, x, w, d, y), yv in zip(layers, eager):
        Nl = w[0].shape[0]
        cols = _cols(Nl, 64, seed=Nl)
        if fmt == "fp8":
            y_ref, l1 = oracle.fp8_linear(x, w[0], w[1], cols=cols)
        else:
            y_ref, l1 = oracle.nvfp4_linear(x, w[0], w[1], w[2], cols=cols)
        check(yv[:, cols], y_ref, l1, True, f"stack {name}")
    cols = _cols(N, 64, seed=3)
    y_ref, l1 = oracle.nvfp4_linear(hx, hw[0], hw[1], hw[2], cols=cols)
    check(eager[-2][:, cols], y_ref, l1, False, "stack lm_head")


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
@pytest.mark.parametrize("M", [1, 4, 8])
def test_back_to_back_bitwise(sk, fmt, M):
    """down (K=17408, N=5120) launched right after gate_up, with PDL, 60 times
    with a poisoned output: every result equals the first bitwise (split-K
    sums run in a fixed order, so any difference is a race), and the first
    matches the oracle on sampled columns.  Guards the ring-stage release and
    the split-K publish order, which a race breaks only now and then."""
    import torch

    (_, Kg, Ng), (_, Kd, Nd) = SHAPES[2], SHAPES[3]
    xs, ws, ds = [], [], []
    for K, N in ((Kg, Ng), (Kd, Nd)):
        x = synth.x_f16(M, K, seed=K + 7)
        w = _f8(N, K, N + 7) if fmt == "fp8" else _nv(N, K, N + 7)
        xs.append(x)
        ws.append(w)
        ds.append((dev(x), dev(w[0]), dev(w[1])))
    yg = torch.empty((M, Ng), dtype=torch.float16, device="cuda:0")
    yd = torch.empty((M, Nd), dtype=torch.float16, device="cuda:0")

    def call(d, w, y):
        if fmt == "fp8":
            sk.fp8_gemm(d[0], d[1], d[2], y=y, f16_out=True)
        else:
            sk.nvfp4_gemm(d[0], d[1], d[2], float(w[2]), y=y, f16_out=True)

    s = torch.cuda.Stream()
    first, bad = None, []
    for it in range(60):
        with torch.cuda.stream(s):
            yd.fill_(float("nan"))
            call(ds[0], ws[0], yg)
            call(ds[1], ws[1], yd)
        s.synchronize()
        got = host(yd)
        if first is None:
            first = got
        elif not np.array_equal(got, first):
            bad.append((it, int(np.sum(~(got == first)))))
    assert not bad, f"results differ from the first run: {bad[:8]}"
    cols = _cols(Nd, 64, seed=Nd + M)
    if fmt == "fp8":
        y_ref, l1 = oracle.fp8_linear(xs[1], ws[1][0], ws[1][1], cols=cols)
    else:
        y_ref, l1 = oracle.nvfp4_linear(xs[1], ws[1][0], ws[1][1], ws[1][2], cols=cols)
    check(first[:, cols], y_ref, l1, True, f"{fmt} down after gate_up M={M}")


def test_lm_head_verify_full_size(sk):
    """The k = 7 verify round on the full vocabulary (K=5120, N=151936, M=8):
    every draft accepted, then the first draft rejected."""
    import torch

    K, N = synth.LM_HEAD_SHAPE
    M = 8
    x = synth.x_f16(M, K, seed=108)
    codes, scales, g = _nv(N, K, 101)
    xd, cd, sd = dev(x), dev(codes), dev(scales)
    _, am = sk.lm_head_argmax(xd, cd, sd, float(g), want_logits=False)
    picks = host(am).astype(np.int64)
    for d in (picks[:7].astype(np.int32), np.concatenate([[int(picks[0] + 1) % N], picks[1:7]]).astype(np.int32)):
        _, am2, acc = sk.lm_head_verify(xd, cd, sd, float(g), torch.from_numpy(d).to("cuda:0"), want_logits=False)
        assert np.array_equal(host(am2), host(am))
        assert tuple(int(v) for v in host(acc)) == oracle.verify(picks, d)
