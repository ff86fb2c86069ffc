"""GPU parity of the NVFP4 lm_head with the fused greedy argmax."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import Guarded, argmax_ok, check, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    import torch

    torch.cuda.set_device(0)
    import fp8_weight_only_skinny_gb300 as skm

    skm.init()
    yield skm
    assert skm.last_device_error() == skm.SK_OK


def _argmax_ok(am, y_ref, l1, logits_gpu):
    """The fused index is the lowest-index max of the same call's FP32 logits
    (bitwise), and agrees with the oracle where its top-2 gap exceeds the bound."""
    argmax_ok(am, y_ref, l1, logits_gpu)


def _guarded_head(sk, x, codes, scales, g, M, N, want_logits=True):
    """lm_head_argmax into guarded logits / argmax buffers; returns host copies."""
    import torch

    lg = Guarded((M, N), torch.float32) if want_logits else None
    am = Guarded((M,), torch.int32, fill=-7)
    sk.lm_head_argmax(dev(x), dev(codes), dev(scales), float(g), logits=lg.t if lg else None, argmax=am.t,
                      want_logits=want_logits)
    return (lg.host("logits") if lg else None), am.host("argmax")


@pytest.mark.parametrize("M", [1, 2, 4, 8])
@pytest.mark.parametrize("K,N", [(1024, 4099), (5120, 3000), (256, 16)])
def test_lm_head_logits_and_argmax(sk, M, K, N):
    x = synth.x_f16(M, K, seed=M * 31 + N)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=N)
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    lg, am = _guarded_head(sk, x, codes, scales, g, M, N)
    check(lg, y_ref, l1, False, "lm_head logits")
    _argmax_ok(am, y_ref, l1, lg)
    # without logits: same indices
    _, am2 = _guarded_head(sk, x, codes, scales, g, M, N, want_logits=False)
    assert np.array_equal(am2, am)


@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("K", [17408, 32768])
def test_lm_head_many_chunks(sk, M, K):
    """17 and 32 k-chunks per row group: the argmax through the owners'
    many-chunk sums (one and two rounds of 24 slots), ragged N."""
    N = 1001
    x = synth.x_f16(M, K, seed=K + M)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=K)
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    lg, am = _guarded_head(sk, x, codes, scales, g, M, N)
    check(lg, y_ref, l1, False, f"lm_head logits K={K}")
    _argmax_ok(am, y_ref, l1, lg)


def test_ties_go_to_the_lowest_index(sk):
    M, K, N = 8, 1024, 700
    x = synth.x_f16(M, K, seed=5)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=5)
    y_ref, _ = oracle.nvfp4_linear(x, codes, scales, g)
    # copy each row's winner to a later and an earlier row: the earliest copy wins
    win = oracle.argmax_rows(y_ref)
    codes2, scales2 = codes.copy(), scales.copy()
    for m in range(M):
        for dst in (3 + 80 * m, N - 1 - m):
            codes2[dst], scales2[dst] = codes[win[m]], scales[win[m]]
    y2, _ = oracle.nvfp4_linear(x, codes2, scales2, g)
    logits, am = sk.lm_head_argmax(dev(x), dev(codes2), dev(scales2), float(g))
    lg, am = host(logits), host(am)
    for m in range(M):
        assert am[m] == int(np.argmax(lg[m]))
        assert lg[m, am[m]] == lg[m].max()


def test_repeated_argmax_is_stable(sk):
    M, K, N = 8, 2048, 9001
    x = synth.x_f16(M, K, seed=9)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=9)
    first = None
    for _ in range(5):
        logits, am = sk.lm_head_argmax(dev(x), dev(codes), dev(scales), float(g))
        cur = (host(logits), host(am))
        if first is None:
            first = cur
        assert np.array_equal(cur[0], first[0]) and np.array_equal(cur[1], first[1])


@pytest.mark.parametrize("var", ["auto", "simt"])
@pytest.mark.parametrize("M", [1, 2, 5, 8])
def test_verify_round(sk, M, var):
    """lm_head_verify: the accepted count and bonus token equal the oracle's
    greedy verification of the same call's picks, for a first rejected draft at
    every position and for every draft accepted; the picks and logits equal
    lm_head_argmax's bitwise and meet the oracle contract."""
    import torch
    from gpu_util import variant

    K, N = 2048, 3001
    x = synth.x_f16(M, K, seed=300 + M)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=301)
    xd, cd, sd = dev(x), dev(codes), dev(scales)
    with variant(sk, var if M == 1 else "auto"):
        lg0, am0 = sk.lm_head_argmax(xd, cd, sd, float(g))
        picks = host(am0).astype(np.int64)
        y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
        _argmax_ok(picks, y_ref, l1, host(lg0))
        cases = []
        for L in range(M):                             # drafts accepted up to L, then one rejected
            d = picks[:M - 1].astype(np.int32).copy()
            if L < M - 1:
                d[L] = (d[L] + 1) % N
            cases.append(d)
        for d in cases:
            dd = torch.from_numpy(np.ascontiguousarray(d) if d.size else np.zeros(1, np.int32)).to("cuda:0")
            glg = Guarded((M, N), torch.float32)
            gam = Guarded((M,), torch.int32, fill=-7)
            gacc = Guarded((2,), torch.int32, fill=-7)
            sk.lm_head_verify(xd, cd, sd, float(g), dd, logits=glg.t, argmax=gam.t, accept=gacc.t)
            lg, am, acc = glg.host("logits"), gam.host("argmax"), gacc.host("accept")
            assert np.array_equal(am, host(am0)) and np.array_equal(lg, host(lg0))
            a, bonus = oracle.verify(picks, d)
            assert tuple(int(v) for v in acc) == (a, bonus), (d, acc, (a, bonus))
