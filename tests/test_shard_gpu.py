"""GPU parity at the pages' per-rank shapes: the 27B decoder's linears split
4-way tensor parallel (qkv, gate_up, lm_head over N; o_proj, down over K), each
rank's shard cut on block boundaries by fp8_weight_only_skinny_gb300.shard.

Column-parallel shards reproduce the full call's rows bitwise (same K, same
kernel variant, so the same per-row summation order); row-parallel shards add
up to the full call within twice the accuracy bound; every shard meets the
oracle contract on sampled columns."""
import functools

import numpy as np
import pytest

import oracle
import synth
from gpu_util import check, dev, host, variant

pytestmark = pytest.mark.gpu

WORLD = 4
TP = [("qkv", 5120, 7168, "n"), ("o_proj", 6144, 5120, "k"), ("gate_up", 5120, 34816, "n"),
      ("down", 17408, 5120, "k")]


@functools.lru_cache(maxsize=None)
def _nv(N, K, seed):
    return synth.nvfp4_weights(N, K, seed=seed)


@functools.lru_cache(maxsize=None)
def _f8(N, K, seed):
    return synth.fp8_weights(N, K, seed=seed)


@pytest.fixture(scope="module")
def sk():
    import torch

    torch.cuda.set_device(0)
    import fp8_weight_only_skinny_gb300 as skm

    skm.init()
    yield skm
    assert skm.last_device_error() == skm.SK_OK


def _cols(N, n=96, seed=0):
    r = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, N // 2, N - 1], r.choice(N, n, replace=False)]))


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
@pytest.mark.parametrize("name,K,N,axis", TP)
@pytest.mark.parametrize("M", [1, 8])
def test_tp4_shards(sk, fmt, name, K, N, axis, M):
    from fp8_weight_only_skinny_gb300 import shard

    x = synth.x_f16(M, K, seed=K + N + M)
    if fmt == "nvfp4":
        codes, scales, g = _nv(N, K, N + 11)
        cut = shard.shard_nvfp4
        run = lambda xx, c, s: host(sk.nvfp4_gemm(dev(xx), dev(c), dev(s), float(g)))
        ref = lambda xx, c, s, cols: oracle.nvfp4_linear(xx, c, s, g, cols=cols)
    else:
        codes, scales = _f8(N, K, N + 12)
        cut = shard.shard_fp8
        run = lambda xx, c, s: host(sk.fp8_gemm(dev(xx), dev(c), dev(s)))
        ref = lambda xx, c, s, cols: oracle.fp8_linear(xx, c, s, cols=cols)
    with variant(sk, "tensor"):               # one variant for the full call and the shards
        full = run(x, codes, scales)
        outs = []
        for r in range(WORLD):
            xs = shard.shard_x(x, axis, r, WORLD)
            cs, ss = cut(codes, scales, axis, r, WORLD)
            y = run(xs, cs, ss)
            outs.append(y)
            if r in (0, WORLD - 1):           # the per-rank shape itself against the oracle
                cols = _cols(y.shape[1], seed=r)
                y_ref, l1 = ref(xs, cs, ss, cols)
                check(y[:, cols], y_ref, l1, False, f"{name} {fmt} rank {r}")
    if axis == "n":
        assert np.array_equal(np.hstack(outs), full)
    else:
        cols = _cols(N, seed=7)
        y_ref, l1 = ref(x, codes, scales, cols)
        total = np.sum(outs, axis=0)
        assert np.all(np.abs(total[:, cols] - full[:, cols]) <= 2 * oracle.tolerance(l1))


@pytest.mark.parametrize("M", [1, 8])
def test_tp4_lm_head_shards(sk, M):
    """The vocabulary split 4 ways: each rank's logits equal the full call's
    bitwise, and the global greedy pick (the max over the ranks' picks, ties to
    the lower rank) equals the full call's argmax."""
    from fp8_weight_only_skinny_gb300 import shard

    K, N = synth.LM_HEAD_SHAPE
    x = synth.x_f16(M, K, seed=50 + M)
    codes, scales, g = _nv(N, K, 101)
    xd = dev(x)
    with variant(sk, "tensor"):
        lg, am = sk.lm_head_argmax(xd, dev(codes), dev(scales), float(g))
        lg, am = host(lg), host(am)
        best = np.full(M, -np.inf)
        pick = np.zeros(M, np.int64)
        for r in range(WORLD):
            cs, ss = shard.shard_nvfp4(codes, scales, "n", r, WORLD)
            lr, ar = sk.lm_head_argmax(xd, dev(cs), dev(ss), float(g))
            lr, ar = host(lr), host(ar)
            n0 = r * (N // WORLD)
            assert np.array_equal(lr, lg[:, n0:n0 + N // WORLD])
            for m in range(M):
                if lr[m, ar[m]] > best[m]:
                    best[m], pick[m] = lr[m, ar[m]], n0 + ar[m]
    assert np.array_equal(pick, am)
