"""GPU parity: the CUDA path against the CPU oracle, element by element.

Every case runs through the C ABI (via the ctypes binding) on seeded synthetic
inputs and compares with the oracle under the accuracy contract
|y - y_ref| <= 1e-3 * sum|x*w| + 1e-6 (+ one FP16 ulp for FP16 output).
Exact cases (identity, one-hot, single-product decodes) are compared bitwise.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import Guarded, check, dev, host, variant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    import torch

    torch.cuda.set_device(0)
    import fp8_weight_only_skinny_gb300 as skm

    skm.init()
    yield skm
    assert skm.last_device_error() == skm.SK_OK


def _out(M, N, f16):
    import torch

    return Guarded((M, N), torch.float16 if f16 else torch.float32)


def nv_run(sk, x, codes, scales, g, f16=False):
    """nvfp4_gemm into an output between guard bands (checked after the call)."""
    y = _out(x.shape[0], codes.shape[0], f16)
    sk.nvfp4_gemm(dev(x), dev(codes), dev(scales), float(g), y=y.t, f16_out=f16)
    return y.host("nvfp4_gemm output")


def f8_run(sk, x, codes, scales, f16=False):
    """fp8_gemm into an output between guard bands (checked after the call)."""
    y = _out(x.shape[0], codes.shape[0], f16)
    sk.fp8_gemm(dev(x), dev(codes), dev(scales), y=y.t, f16_out=f16)
    return y.host("fp8_gemm output")


# ------------------------------------------------------------ config C0 ---

@pytest.mark.parametrize("f16", [False, True])
def test_c0_gemv_k512_n256(sk, f16):
    x = synth.x_f16(1, 512, seed=0)
    codes, scales, g = synth.nvfp4_weights(256, 512, seed=0)
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    check(nv_run(sk, x, codes, scales, g, f16), y_ref, l1, f16, "C0")


# ------------------------------------------- multi-tile, ragged, all M ---

NV_SHAPES = [(256, 1), (256, 17), (1024, 16), (1280, 100), (3072, 257), (2304, 33), (5120, 40)]


@pytest.mark.parametrize("K,N", NV_SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
def test_nvfp4_ragged_shapes(sk, K, N, M):
    x = synth.x_f16(M, K, seed=K + N + M)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=K * 7 + N)
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    check(nv_run(sk, x, codes, scales, g), y_ref, l1, False, f"nvfp4 M{M} K{K} N{N}")
    check(nv_run(sk, x, codes, scales, g, True), y_ref, l1, True, f"nvfp4 f16 M{M} K{K} N{N}")


F8_SHAPES = [(128, 1), (384, 17), (1024, 128), (1152, 129), (2048, 300), (3200, 40)]


@pytest.mark.parametrize("K,N", NV_SHAPES)
@pytest.mark.parametrize("var", ["simt", "tensor"])
def test_nvfp4_ragged_shapes_one_token_variants(sk, K, N, var):
    """M = 1 through each kernel variant explicitly (the automatic choice
    depends on the shape)."""
    x = synth.x_f16(1, K, seed=K + N + 11)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=K * 7 + N)
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    with variant(sk, var):
        check(nv_run(sk, x, codes, scales, g), y_ref, l1, False, f"nvfp4 {var} K{K} N{N}")
        check(nv_run(sk, x, codes, scales, g, True), y_ref, l1, True, f"nvfp4 f16 {var} K{K} N{N}")


@pytest.mark.parametrize("K,N", F8_SHAPES)
@pytest.mark.parametrize("var", ["simt", "tensor"])
def test_fp8_ragged_shapes_one_token_variants(sk, K, N, var):
    x = synth.x_f16(1, K, seed=K + N + 12)
    codes, scales = synth.fp8_weights(N, K, seed=K * 5 + N)
    y_ref, l1 = oracle.fp8_linear(x, codes, scales)
    with variant(sk, var):
        check(f8_run(sk, x, codes, scales), y_ref, l1, False, f"fp8 {var} K{K} N{N}")
        check(f8_run(sk, x, codes, scales, True), y_ref, l1, True, f"fp8 f16 {var} K{K} N{N}")


@pytest.mark.parametrize("K,N", F8_SHAPES)
@pytest.mark.parametrize("M", [1, 2, 4, 6, 8])
def test_fp8_ragged_shapes(sk, K, N, M):
    x = synth.x_f16(M, K, seed=K + N + M + 1)
    codes, scales = synth.fp8_weights(N, K, seed=K * 5 + N)
    y_ref, l1 = oracle.fp8_linear(x, codes, scales)
    check(f8_run(sk, x, codes, scales), y_ref, l1, False, f"fp8 M{M} K{K} N{N}")
    check(f8_run(sk, x, codes, scales, True), y_ref, l1, True, f"fp8 f16 M{M} K{K} N{N}")


ONE_AND_EIGHT = [(1, "simt"), (1, "tensor"), (8, "auto")]


@pytest.mark.parametrize("M,var", ONE_AND_EIGHT)
def test_long_k_many_partials(sk, M, var):
    """K = 17408 gives 17 k-chunks per row group: the split-K fix-up path."""
    K, N = 17408, 48
    x = synth.x_f16(M, K, seed=21)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=21)
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    c8, s8 = synth.fp8_weights(N, K, seed=22)
    f_ref, fl1 = oracle.fp8_linear(x, c8, s8)
    with variant(sk, var):
        check(nv_run(sk, x, codes, scales, g), y_ref, l1, False, "nvfp4 long K")
        check(f8_run(sk, x, c8, s8), f_ref, fl1, False, "fp8 long K")


@pytest.mark.parametrize("M,var", ONE_AND_EIGHT)
@pytest.mark.parametrize("K", [32768, 49408])
def test_very_long_k_several_fixup_rounds(sk, K, M, var):
    """32 and 49 k-chunks per row group (the last one ragged at K = 49408):
    the owners sum the partial slots of a row group in rounds of 24 chunks, so
    these take two and three rounds; N = 77 leaves a ragged row group."""
    N = 77
    x = synth.x_f16(M, K, seed=23)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=23)
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    c8, s8 = synth.fp8_weights(N, K, seed=24)
    f_ref, fl1 = oracle.fp8_linear(x, c8, s8)
    with variant(sk, var):
        check(nv_run(sk, x, codes, scales, g), y_ref, l1, False, f"nvfp4 K={K}")
        check(f8_run(sk, x, c8, s8), f_ref, fl1, False, f"fp8 K={K}")


# ------------------------------------------------- exact / bitwise cases ---

@pytest.mark.parametrize("M,var", ONE_AND_EIGHT)
def test_identity_is_bitwise(sk, M, var):
    with variant(sk, var):
        _identity_case(sk, M)


def _identity_case(sk, M):
    K = N = 512
    x = synth.x_f16(M, K, seed=31)
    nib = np.zeros((N, K), np.uint8)
    nib[np.arange(N), np.arange(K)] = 0x2
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    scales = np.full((N, K // 16), 0x38, np.uint8)
    assert np.array_equal(nv_run(sk, x, codes, scales, 1.0), x.astype(np.float64))
    assert np.array_equal(nv_run(sk, x, codes, scales, 1.0, True), x.astype(np.float64))
    c8 = np.zeros((N, K), np.uint8)
    c8[np.arange(N), np.arange(K)] = 0x38
    s8 = np.ones((4, 4), np.float32)
    assert np.array_equal(f8_run(sk, x, c8, s8), x.astype(np.float64))


@pytest.mark.parametrize("M,var", ONE_AND_EIGHT + [(4, "auto")])
def test_every_code_byte_decodes_exactly(sk, M, var):
    """Row n holds code byte n at k = (0, 1) and scale code 0x38: y[m][n] =
    x[m][0]*E2M1(n & 15) + x[m][1]*E2M1(n >> 4), a sum of two exact products with
    x[1] = 1024*x[0] (powers of two), so the result is exact."""
    K, N = 1024, 256
    x = np.zeros((M, K), np.float16)
    x[:, 0] = np.float16(0.5) * (np.arange(M) + 1)
    x[:, 1] = x[:, 0] * np.float16(1024)
    codes = np.zeros((N, K // 2), np.uint8)
    codes[:, 0] = np.arange(256)
    scales = np.full((N, K // 16), 0x38, np.uint8)
    y_ref, _ = oracle.nvfp4_linear(x, codes, scales, 1.0)
    with variant(sk, var):
        assert np.array_equal(nv_run(sk, x, codes, scales, 1.0), y_ref)


@pytest.mark.parametrize("M,var", ONE_AND_EIGHT)
def test_every_scale_code_decodes_exactly(sk, M, var):
    """Row n: code 1.0 at k = 0 and block scale code n (NaN codes give NaN)."""
    K, N = 256, 256
    x = np.zeros((M, K), np.float16)
    x[:, 0] = np.float16(1.0)
    codes = np.zeros((N, K // 2), np.uint8)
    codes[:, 0] = 0x02
    scales = np.zeros((N, K // 16), np.uint8)
    scales[:, 0] = np.arange(256)
    y_ref, _ = oracle.nvfp4_linear(x, codes, scales, 1.0)
    with variant(sk, var):
        y = nv_run(sk, x, codes, scales, 1.0)
    nan = np.isnan(y_ref)
    assert np.array_equal(np.isnan(y), nan)
    assert np.array_equal(y[~nan], y_ref[~nan])


@pytest.mark.parametrize("M,var", ONE_AND_EIGHT)
def test_every_fp8_code_decodes_exactly(sk, M, var):
    K, N = 128, 256
    x = np.zeros((M, K), np.float16)
    x[:, 5] = np.float16(1.0)
    codes = np.zeros((N, K), np.uint8)
    codes[:, 5] = np.arange(256)
    s8 = np.array([[2.0], [0.5]], np.float32)
    y_ref, _ = oracle.fp8_linear(x, codes, s8)
    with variant(sk, var):
        y = f8_run(sk, x, codes, s8)
    nan = np.isnan(y_ref)
    assert np.array_equal(np.isnan(y), nan)
    assert np.array_equal(y[~nan], y_ref[~nan])


@pytest.mark.parametrize("k0", [0, 1, 15, 16, 31, 32, 255, 511, 1023, 1024, 1025, 2047])
def test_one_hot_positions_bitwise(sk, k0):
    M, N, K = 8, 40, 2048
    x = synth.x_f16(M, K, seed=k0)
    for n0, c in ((0, 0x7), (17, 0xB), (39, 0x3)):
        nib = np.zeros((N, K), np.uint8)
        nib[n0, k0] = c
        codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
        scales = (0x20 + (np.arange(N * (K // 16)) % 48)).astype(np.uint8).reshape(N, K // 16)
        y_ref, _ = oracle.nvfp4_linear(x, codes, scales, np.float32(0.25))
        for mm in (1, 2, 4, 8):
            y = nv_run(sk, x[:mm], codes, scales, np.float32(0.25))
            assert np.array_equal(y, y_ref[:mm]), (k0, n0, mm)
        with variant(sk, "simt"):
            y = nv_run(sk, x[:1], codes, scales, np.float32(0.25))
        assert np.array_equal(y, y_ref[:1]), (k0, n0, "simt")


# --------------------------------------------------------- invariants -----

def test_power_of_two_scaling_and_gscale_bitwise(sk):
    M, K, N = 8, 3072, 96
    x = synth.x_f16(M, K, seed=41)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=41)
    for mm in (1, 8):
        y = nv_run(sk, x[:mm], codes, scales, g)
        y4 = nv_run(sk, (x[:mm].astype(np.float32) * 4).astype(np.float16), codes, scales, g)
        assert np.array_equal(y4, 4 * y)
        y2 = nv_run(sk, x[:mm], codes, scales, np.float32(2 * g))
        assert np.array_equal(y2, 2 * y)


def test_repeated_calls_are_bitwise_identical(sk):
    M, K, N = 8, 6144, 200
    x = synth.x_f16(M, K, seed=51)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=51)
    c8, s8 = synth.fp8_weights(N, K, seed=51)
    for mm in (1, 8):
        first = nv_run(sk, x[:mm], codes, scales, g)
        f_first = f8_run(sk, x[:mm], c8, s8)
        for _ in range(9):
            assert np.array_equal(nv_run(sk, x[:mm], codes, scales, g), first)
            assert np.array_equal(f8_run(sk, x[:mm], c8, s8), f_first)


def test_rows_independent_within_a_variant(sk):
    """Rows of an M-row call equal the same rows run alone on the same kernel
    variant bitwise (the MMA variant is forced for the single rows)."""
    M, K, N = 8, 2048, 64
    x = synth.x_f16(M, K, seed=61)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=61)
    c8, s8 = synth.fp8_weights(N, K, seed=61)
    y8 = nv_run(sk, x, codes, scales, g)
    f8 = f8_run(sk, x, c8, s8)
    prev = sk.set_variant(sk.VARIANT_TENSOR)
    try:
        for m in range(M):
            assert np.array_equal(nv_run(sk, x[m:m + 1], codes, scales, g)[0], y8[m])
            assert np.array_equal(f8_run(sk, x[m:m + 1], c8, s8)[0], f8[m])
        # across variants (SIMT for one row vs MMA for eight) within twice the bound
        sk.set_variant(sk.VARIANT_SIMT)
        y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
        for m in range(M):
            y1 = nv_run(sk, x[m:m + 1], codes, scales, g)[0]
            assert np.all(np.abs(y1 - y8[m]) <= 2 * oracle.tolerance(l1[m]))
    finally:
        sk.set_variant(prev)


@pytest.mark.parametrize("M", [4, 8])
def test_activation_alignment_does_not_change_results(sk, M):
    """From M = 4 the tensor-core variant loads 32-byte aligned activations 32
    bytes per lane, else 16: x at a 32-byte boundary and x 16 bytes past one
    give bitwise the same outputs (both formats, FP32 and FP16 output, one
    k-chunk and several), and the aligned ones match the oracle."""
    import torch

    for K, N in ((1024, 64), (5120, 200)):
        x = synth.x_f16(M, K, seed=71 + K)
        codes, scales, g = synth.nvfp4_weights(N, K, seed=71)
        c8, s8 = synth.fp8_weights(N, K, seed=71)
        cd, sd, c8d, s8d = dev(codes), dev(scales), dev(c8), dev(s8)
        outs = []
        for off in (0, 8):                      # halves: 0 or 16 bytes past the boundary
            buf = torch.zeros(M * K + 16, dtype=torch.float16, device="cuda:0")
            assert buf.data_ptr() % 32 == 0
            xd = buf[off:off + M * K].view(M, K)
            xd.copy_(dev(x))
            assert (xd.data_ptr() % 32 == 0) == (off == 0)
            got = []
            for f16 in (False, True):
                y = _out(M, N, f16)
                sk.nvfp4_gemm(xd, cd, sd, float(g), y=y.t, f16_out=f16)
                got.append(y.host("nvfp4_gemm output"))
                y = _out(M, N, f16)
                sk.fp8_gemm(xd, c8d, s8d, y=y.t, f16_out=f16)
                got.append(y.host("fp8_gemm output"))
            outs.append(got)
        for a, b in zip(*outs):
            assert np.array_equal(a, b)
        y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
        check(outs[0][0], y_ref, l1, False, f"nvfp4 aligned x M{M} K{K}")
        y_ref, l1 = oracle.fp8_linear(x, c8, s8)
        check(outs[0][1], y_ref, l1, False, f"fp8 aligned x M{M} K{K}")


# ------------------------------------------------------ degenerate cases ---

def test_k_zero_gives_zeros_and_n_zero_is_a_noop(sk):
    import torch

    x = torch.zeros((3, 0), dtype=torch.float16, device="cuda:0")
    codes = torch.zeros((5, 0), dtype=torch.uint8, device="cuda:0")
    scales = torch.zeros((5, 0), dtype=torch.uint8, device="cuda:0")
    # tensors of zero elements have null data pointers: pass aligned dummies
    buf = torch.zeros(64, dtype=torch.uint8, device="cuda:0")
    y = torch.full((3, 5), 7.0, device="cuda:0")
    st = sk.lib.nvfp4_gemm(buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), 1.0, y.data_ptr(), 3, 5, 0, None)
    torch.cuda.synchronize()
    assert st == 0 and torch.all(y == 0)
    y.fill_(7.0)
    st = sk.lib.fp8_gemm(buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), y.data_ptr(), 3, 0, 128, None)
    torch.cuda.synchronize()
    assert st == 0 and torch.all(y == 7.0)
    del x, codes, scales


def test_workspace_too_small_is_reported(sk):
    import torch

    sk.init(64 << 10)             # the control block and 60 KiB of partial-sum slots
    try:
        x = dev(synth.x_f16(8, 5120, seed=1))
        codes, scales, g = synth.nvfp4_weights(4096, 5120, seed=1)
        c, s = dev(codes), dev(scales)
        y = torch.empty((8, 4096), device="cuda:0")
        st = sk.lib.nvfp4_gemm(x.data_ptr(), c.data_ptr(), s.data_ptr(), float(g), y.data_ptr(),
                               8, 4096, 5120, None)
        assert st == 7
    finally:
        sk.init()


def test_bounded_wait_times_out_and_context_survives(sk):
    """Failure injection: the next kernel's producer issues no copies, so its
    consumers' bounded waits run out; the kernel still finishes and reports
    SK_ERR_TIMEOUT, and the next normal call is correct."""
    M, K, N = 1, 1024, 64
    x = synth.x_f16(M, K, seed=2)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=2)
    sk.lib.sk_inject_wait_timeout(1)
    nv_run(sk, x, codes, scales, g)
    assert sk.last_device_error() == 6
    assert sk.last_device_error() == 0          # the word was cleared
    sk.init()
    y_ref, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    check(nv_run(sk, x, codes, scales, g), y_ref, l1, False, "after timeout")
