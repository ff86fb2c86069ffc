"""GPU parity of the sampled lm_head pick (lm_head_sample) against the oracle
(oracle/sample.py) applied to the same call's FP32 logits: the picks agree
wherever the draw and the top-p cut are farther than FP32 rounding from a
boundary, and otherwise the pick is still a kept candidate."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import dev, host

pytestmark = pytest.mark.gpu

SETTINGS = [(0.6, 50, 0.9), (1.0, 1024, 1.0), (0.0, 10, 1.0), (2.0, 1, 1.0), (0.8, 300, 0.5), (1.3, 7, 0.99)]


@pytest.fixture(scope="module")
def sk():
    import torch

    torch.cuda.set_device(0)
    import fp8_weight_only_skinny_gb300 as skm

    skm.init()
    yield skm
    assert skm.last_device_error() == skm.SK_OK


def _check_picks(tok, logits, u, T, k, p):
    for m in range(logits.shape[0]):
        want = oracle.sample_row(logits[m], u[m], T, k, p)
        if tok[m] == want:
            continue
        assert oracle.sample_margin(logits[m], u[m], T, k, p) < 1e-5, (m, tok[m], want)
        order = sorted(range(logits.shape[1]), key=lambda i: (-float(logits[m, i]), i))[:k]
        assert tok[m] in order, (m, tok[m])


@pytest.mark.parametrize("T,k,p", SETTINGS)
@pytest.mark.parametrize("M,N", [(1, 3001), (8, 3001), (4, 151936)])
def test_sampled_pick_matches_the_oracle(sk, M, N, T, k, p):
    import torch

    K = 2048 if N < 100000 else 5120
    x = synth.x_f16(M, K, seed=M + N)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=17 if N < 100000 else 101)
    r = np.random.default_rng(M * 7 + k)
    u = r.random(M).astype(np.float32)
    u[0] = 0.0
    if M > 1:
        u[1] = np.float32(0.999999)
    lg, tok = sk.lm_head_sample(dev(x), dev(codes), dev(scales), float(g), torch.from_numpy(u).to("cuda:0"),
                                T, k, p)
    logits, tok = host(lg).astype(np.float32), host(tok)
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g, cols=np.arange(0, N, 97))
    assert np.all(np.abs(logits[:, ::97] - y_ref) <= oracle.tolerance(l1))     # the logits themselves
    _check_picks(tok, logits, u, T, k, p)


@pytest.mark.parametrize("M,N,K,T,k,p", [(2, 400000, 256, 0.6, 50, 0.9), (2, 400000, 256, 1.0, 1024, 1.0),
                                          (3, 5, 256, 1.0, 5, 1.0), (3, 5, 256, 0.0, 3, 1.0),
                                          (1, 9, 256, 0.9, 9, 0.8)])
def test_row_lengths_at_the_slice_limits(sk, M, N, K, T, k, p):
    """A row is split over a cluster of CTAs, each keeping up to 49152 keys in
    shared memory: rows longer than that per CTA (the rest re-read), and rows
    shorter than the cluster (CTAs with no keys at all)."""
    import torch

    x = synth.x_f16(M, K, seed=N + k)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=23)
    u = np.random.default_rng(N + k).random(M).astype(np.float32)
    lg, tok = sk.lm_head_sample(dev(x), dev(codes), dev(scales), float(g), torch.from_numpy(u).to("cuda:0"),
                                T, k, p)
    _check_picks(host(tok), host(lg).astype(np.float32), u, T, k, p)


@pytest.mark.parametrize("T,k,p", [(1.0, 40, 1.0), (0.0, 12, 1.0), (0.7, 20, 0.6)])
@pytest.mark.parametrize("N", [700, 7000])
def test_ties_are_broken_by_the_lower_index(sk, N, T, k, p):
    """Rows n and n + 7j of the weight are equal, so the logits tie in groups
    of many, spread over every CTA of a row's cluster: the candidates must
    come in index order within a tie."""
    import torch

    M, K = 8, 1024
    x = synth.x_f16(M, K, seed=3)
    base, scales_b, g = synth.nvfp4_weights(7, K, seed=4)
    codes = np.ascontiguousarray(np.tile(base, (N // 7, 1)))
    scales = np.ascontiguousarray(np.tile(scales_b, (N // 7, 1)))
    u = np.linspace(0.0, 0.99, M).astype(np.float32)
    lg, tok = sk.lm_head_sample(dev(x), dev(codes), dev(scales), float(g), torch.from_numpy(u).to("cuda:0"),
                                T, k, p)
    _check_picks(host(tok), host(lg).astype(np.float32), u, T, k, p)
