"""GPU parity of the weight quantizers: bit-exact against the oracle
(oracle/quant.py) on random, extreme and exactly-tied inputs, and the
quantized weights feed the linear layers like any others."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import check, dev, host

pytestmark = pytest.mark.gpu

F16 = np.float16


@pytest.fixture(scope="module")
def sk():
    import torch

    torch.cuda.set_device(0)
    import fp8_weight_only_skinny_gb300 as skm

    skm.init()
    yield skm
    assert skm.last_device_error() == skm.SK_OK


def _weights(N, K, seed, kind):
    r = np.random.default_rng(seed)
    if kind == "normal":
        return (r.standard_normal((N, K)) * 0.02).astype(F16)
    if kind == "wide":          # every FP16 magnitude class, both signs, zeros and subnormals
        e = r.integers(-24, 15, size=(N, K)).astype(np.float64)             # finite: below 2^15
        w = (r.uniform(1, 1.99, size=(N, K)) * np.exp2(e) * r.choice([-1, 1], size=(N, K))).astype(F16)
        assert np.all(np.isfinite(w))
        w.flat[r.choice(w.size, w.size // 20, replace=False)] = 0
        w.flat[r.choice(w.size, w.size // 20, replace=False)] = -0.0
        w.flat[:4] = [65504, -65504, 6e-8, -6e-8]
        return w
    raise ValueError(kind)


@pytest.mark.parametrize("N,K", [(128, 128), (256, 1024), (300, 200), (77, 1032)])
@pytest.mark.parametrize("kind", ["normal", "wide"])
def test_fp8_quantize_bitexact(sk, N, K, kind):
    w = _weights(N, K, N * K, kind)
    codes, scales = sk.fp8_quantize(dev(w))
    c_ref, s_ref = oracle.quantize_fp8(w)
    assert np.array_equal(host(scales).astype(np.float32), s_ref)
    got = host(codes)
    assert np.array_equal(got, c_ref), int(np.sum(got != c_ref))


@pytest.mark.parametrize("N,K", [(16, 256), (300, 512), (77, 1040), (1, 16)])
@pytest.mark.parametrize("kind", ["normal", "wide"])
def test_nvfp4_quantize_bitexact(sk, N, K, kind):
    w = _weights(N, K, N + K, kind)
    codes, scales, g = sk.nvfp4_quantize(dev(w))
    c_ref, s_ref, g_ref = oracle.quantize_nvfp4(w)
    assert np.float32(host(g)[0]) == g_ref
    assert np.array_equal(host(scales), s_ref)
    got = host(codes)
    assert np.array_equal(got, c_ref), int(np.sum(got != c_ref))


def test_fp8_all_zero_block(sk):
    """An all-zero 128 x 128 block: scale 1 and zero codes (signs kept), as the oracle."""
    w = (np.random.default_rng(9).standard_normal((256, 384)) * 0.02).astype(F16)
    w[128:, 128:256] = 0
    w[130, 131] = -0.0
    codes, scales = sk.fp8_quantize(dev(w))
    c_ref, s_ref = oracle.quantize_fp8(w)
    assert s_ref[1, 1] == 1.0
    assert np.array_equal(host(scales).astype(np.float32), s_ref)
    assert np.array_equal(host(codes), c_ref)


def _full_size_weight():
    """One FP16 weight of the gate_up shape (34816 x 5120) the benchmark times,
    N(0, 0.02) with a few extremes planted in known places."""
    N, K = 34816, 5120
    w = (np.random.default_rng(91).standard_normal((N, K), dtype=np.float32) * 0.02).astype(F16)
    w[0, :4] = [0.5, -0.75, 0.0, -0.0]
    w[N - 1, K - 16:] = 0                       # an all-zero 16-block in the last row
    w[12345, 678] = -3.0                        # the tensor maximum
    return w


def test_fp8_quantize_full_size_sampled_blocks(sk):
    """The full gate_up weight through the GPU quantizer, 48 of its 128 x 128
    blocks (corners included) checked bitwise against the oracle."""
    w = _full_size_weight()
    N, K = w.shape
    codes, scales = sk.fp8_quantize(dev(w))
    codes, scales = host(codes), host(scales).astype(np.float32)
    nb, kb = N // 128, K // 128
    r = np.random.default_rng(5)
    blocks = {(0, 0), (nb - 1, kb - 1), (0, kb - 1), (nb - 1, 0), (96, 5)}
    while len(blocks) < 48:
        blocks.add((int(r.integers(nb)), int(r.integers(kb))))
    for i, j in sorted(blocks):
        blk = w[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
        c_ref, s_ref = oracle.quantize_fp8(blk)
        assert scales[i, j] == s_ref[0, 0], (i, j)
        assert np.array_equal(codes[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128], c_ref), (i, j)


def test_nvfp4_quantize_full_size_sampled_rows(sk):
    """The full gate_up weight through the GPU quantizer: the tensor scale, and
    64 sampled rows (first, last, the maximum's) bitwise against the oracle
    given the whole tensor's maximum."""
    w = _full_size_weight()
    N, K = w.shape
    codes, scales, g = sk.nvfp4_quantize(dev(w))
    amax = np.float32(np.max(np.abs(w.astype(np.float32))))
    rows = np.unique(np.concatenate([[0, 12345, N - 1], np.random.default_rng(6).choice(N, 61, replace=False)]))
    c_ref, s_ref, g_ref = oracle.quantize_nvfp4(w[rows], amax=amax)
    assert np.float32(host(g)[0]) == g_ref == np.float32(np.float32(3.0) / np.float32(2688.0))
    assert np.array_equal(host(scales)[rows], s_ref)
    assert np.array_equal(host(codes)[rows], c_ref)


def test_exact_ties_round_to_even(sk):
    # FP8: a block whose maximum is 448 has scale 1, so w / s is w itself; the
    # midpoints between neighbouring E4M3 values that FP16 holds exactly are ties.
    vals = oracle.e4m3_to_f64(np.arange(0x7F))
    mids = (vals[:-1] + vals[1:]) / 2
    mids = mids[mids.astype(F16).astype(np.float64) == mids]
    w = np.zeros((128, 128), F16)
    w[0, 0] = 448
    w.flat[1:1 + mids.size] = mids
    w.flat[200:200 + mids.size] = -mids
    codes, scales = sk.fp8_quantize(dev(w))
    assert np.array_equal(host(codes), oracle.quantize_fp8(w)[0])
    # NVFP4: tensor maximum 2688 gives G = 1; a block with maximum 6 gets scale 1,
    # so w / (S G) is w itself: the E2M1 midpoints 0.25 ... 5 are ties.
    w = np.zeros((2, 32), F16)
    w[0, 0] = 2688
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], F16)
    w[1, 0:8], w[1, 8:16] = ties, -ties
    codes, scales, g = sk.nvfp4_quantize(dev(w))
    c_ref, s_ref, g_ref = oracle.quantize_nvfp4(w)
    assert g_ref == 1.0 and s_ref[1, 0] == 0x38
    assert np.array_equal(host(codes), c_ref) and np.array_equal(host(scales), s_ref)


def test_nvfp4_quotients_on_the_boundary_grid(sk):
    """Weights whose quotients w / (S G) are exactly E2M1 values or midpoints
    between them (G = 2^-10, every 16-block's scale an exact E4M3 value S): the
    kernel's products land on or next to its boundary grid almost everywhere,
    so nearly every pair takes the division path -- bitwise against the oracle."""
    r = np.random.default_rng(71)
    N, K = 256, 1024
    G = 2.0 ** -10
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5])
    S = oracle.e4m3_to_f64(np.arange(0x08, 0x60))[r.integers(0, 0x58, (N, K // 16))]
    m = r.choice(vals, (N, K // 16, 16)) * r.choice([-1.0, 1.0], (N, K // 16, 16))
    m[:, :, 0] = 6.0                                   # each block's maximum: 6 S G, so its scale is S
    w64 = (m * (S * G)[:, :, None]).reshape(N, K)
    w64[0, :16] = 0.0
    w64[0, 0] = 2688 * G                               # the tensor maximum: G = 2^-10
    w = w64.astype(F16)
    assert np.array_equal(w.astype(np.float64), w64)   # every weight exact in FP16
    codes, scales, g = sk.nvfp4_quantize(dev(w))
    c_ref, s_ref, g_ref = oracle.quantize_nvfp4(w)
    assert g_ref == np.float32(G) and np.float32(host(g)[0]) == g_ref
    assert np.array_equal(host(scales), s_ref)
    got = host(codes)
    assert np.array_equal(got, c_ref), int(np.sum(got != c_ref))


def test_fp8_quotients_on_the_boundary_grid(sk):
    """FP8 blocks whose scale s = max|w| / 448 is 2^-8 times 1, 1.25, 1.5 or 1.75
    and whose weights are s times E4M3 values or midpoints between them (each
    block holding +-448 s): w / s is exact, its product with RN(1/s) sits on or
    next to the boundary grid, and the division path decides -- bitwise against
    the oracle."""
    r = np.random.default_rng(72)
    N, K = 384, 512
    e = oracle.e4m3_to_f64(np.arange(0x7F))
    vals = np.concatenate([e, (e[:-1] + e[1:]) / 2])
    vals = vals[(vals <= 448) & (vals >= 2.0 ** -9)]
    w64 = np.zeros((N, K))
    for i in range(N // 128):
        for j in range(K // 128):
            s = 2.0 ** -8 * r.choice([1.0, 1.25, 1.5, 1.75])
            v = r.choice(vals, (128, 128)) * r.choice([-1.0, 1.0], (128, 128))
            v[0, 0] = 448.0
            w64[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128] = v * s
    w = w64.astype(F16)
    assert np.array_equal(w.astype(np.float64), w64)   # every weight exact in FP16
    codes, scales = sk.fp8_quantize(dev(w))
    c_ref, s_ref = oracle.quantize_fp8(w)
    assert np.array_equal(host(scales).astype(np.float32), s_ref)
    got = host(codes)
    assert np.array_equal(got, c_ref), int(np.sum(got != c_ref))


@pytest.mark.parametrize("M", [1, 8])
def test_quantized_weights_feed_the_linears(sk, M):
    """GPU-quantized weights through nvfp4_gemm / fp8_gemm meet the oracle
    contract on those codes, and the product stays near the FP16 one."""
    K, N = 2048, 384
    w = _weights(N, K, 9, "normal")
    x = synth.x_f16(M, K, seed=9)
    codes, scales, g = sk.nvfp4_quantize(dev(w))
    y = host(sk.nvfp4_gemm(dev(x), codes, scales, float(host(g)[0])))
    y_ref, l1 = oracle.nvfp4_linear(x, host(codes), host(scales), np.float32(host(g)[0]))
    check(y, y_ref, l1, False, "nvfp4 from the GPU quantizer")
    c8, s8 = sk.fp8_quantize(dev(w))
    y8 = host(sk.fp8_gemm(dev(x), c8, s8))
    y8_ref, l18 = oracle.fp8_linear(x, host(c8), host(s8))
    check(y8, y8_ref, l18, False, "fp8 from the GPU quantizer")
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    scale = np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64)).T
    assert np.all(np.abs(y - exact) <= 0.2 * scale)          # 4-bit weights: coarse, but close
    assert np.all(np.abs(y8 - exact) <= 0.07 * scale)        # 8-bit weights: closer


@pytest.mark.parametrize("M", [1, 8])
def test_quantize_then_multiply_on_one_stream(sk, M):
    """fp8_quantize rewrites the codes and scales and fp8_gemm reads them
    right after it on the same stream, with programmatic dependent launch on
    and no synchronisation in between: each product must use the weights just
    written (a linear kernel streams weights before its dependency wait, so the
    library launches the first linear call after a quantizer without PDL).
    Three rounds alternate two weight matrices in the same buffers."""
    import torch

    N, K = 4096, 5120
    ws = [_weights(N, K, seed, "normal") for seed in (61, 62)]
    refs = []
    x = synth.x_f16(M, K, seed=63)
    for w in ws:
        c, s = oracle.quantize_fp8(w)
        refs.append(oracle.fp8_linear(x, c, s))
    wd = [dev(w) for w in ws]
    xd = dev(x)
    codes = torch.empty((N, K), dtype=torch.uint8, device="cuda:0")
    scales = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device="cuda:0")
    ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda:0") for _ in range(3)]
    prev = sk.set_pdl(True)
    try:
        s = torch.cuda.Stream()
        sp = s.cuda_stream
        for r in range(3):
            assert sk.lib.fp8_quantize(wd[r % 2].data_ptr(), codes.data_ptr(), scales.data_ptr(), N, K, sp) == 0
            assert sk.lib.fp8_gemm(xd.data_ptr(), codes.data_ptr(), scales.data_ptr(), ys[r].data_ptr(),
                                   M, N, K, sp) == 0
        s.synchronize()
    finally:
        sk.set_pdl(prev)
    for r in range(3):
        y_ref, l1 = refs[r % 2]
        check(host(ys[r]), y_ref, l1, False, f"fp8 gemm right after quantize, round {r}")
