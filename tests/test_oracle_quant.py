"""Pins of the quantizer oracle (oracle/quant.py) on the CPU.

Rounding is pinned against the formats' own values (every code maps back to
itself), hand-worked ties and saturation, and PyTorch's float8_e4m3fn
conversion (a library routine); the FP8 quantizer against the same rule
written with PyTorch's conversion (synth.fp8_quantize); the NVFP4 quantizer
against closed forms (the tensor maximum becomes +-6 at scale 448, an
all-zero block gets a zero scale and signed zero codes) and its error bound."""
import numpy as np
import pytest

import oracle
import synth

F32 = np.float32


def test_every_e4m3_value_rounds_to_its_own_code():
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue                                            # NaN codes
        v = oracle.e4m3_to_f64(c)[0]
        assert int(oracle.e4m3_round(np.array([v], F32))[0]) == c, hex(c)


def test_e4m3_ties_go_to_the_even_code_and_values_saturate():
    vals = oracle.e4m3_to_f64(np.arange(0x7F))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(F32)
    exact = mids.astype(np.float64) == (vals[:-1] + vals[1:]) / 2   # midpoints representable in f32
    got = oracle.e4m3_round(mids[exact]).astype(int)
    lo = np.arange(0x7E)[exact]
    assert np.all(got == np.where(lo % 2 == 0, lo, lo + 1))
    assert list(oracle.e4m3_round(np.array([1000.0, -1e9, 448.0, 464.0], F32))) == [0x7E, 0xFE, 0x7E, 0x7E]
    assert list(oracle.e4m3_round(np.array([0.0, -0.0, -1e-30], F32))) == [0x00, 0x80, 0x80]


def test_e4m3_rounding_matches_torch_conversion():
    torch = pytest.importorskip("torch")
    r = np.random.default_rng(1)
    v = np.concatenate([r.standard_normal(200000) * 50, r.standard_normal(50000) * 1e-2,
                        r.uniform(-448, 448, 50000)]).astype(F32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_round(v), ref)


def test_e2m1_rounding_table():
    cases = {0.0: 0, 0.24: 0, 0.25: 0, 0.26: 1, 0.5: 1, 0.75: 2, 1.0: 2, 1.25: 2, 1.5: 3, 1.75: 4,
             2.0: 4, 2.5: 4, 2.6: 5, 3.0: 5, 3.5: 6, 4.0: 6, 5.0: 6, 5.1: 7, 6.0: 7, 7.0: 7, 1e9: 7}
    for v, c in cases.items():
        assert int(oracle.e2m1_round(np.array([v], F32))[0]) == c, v
        assert int(oracle.e2m1_round(np.array([-v], F32))[0]) == c | 8, -v
    for c in range(16):
        assert int(oracle.e2m1_round(oracle.e2m1_to_f64(c).astype(F32))[0]) == c


@pytest.mark.parametrize("N,K", [(128, 256), (300, 200), (77, 1024)])
def test_fp8_quantizer_matches_the_torch_rounding_rule(N, K):
    pytest.importorskip("torch")
    w = (np.random.default_rng(N + K).standard_normal((N, K)) * 0.02).astype(np.float16)
    w[0, :5] = [0.0, -0.0, 65504, -65504, 6e-8]
    codes, scales = oracle.quantize_fp8(w)
    c2, s2 = synth.fp8_quantize(w.astype(F32))
    assert np.array_equal(scales, s2)
    assert np.array_equal(codes, c2)


def test_fp8_quantizer_error_bound_and_extremes():
    w = (np.random.default_rng(3).standard_normal((256, 384)) * 0.02).astype(np.float16)
    codes, scales = oracle.quantize_fp8(w)
    deq = oracle.e4m3_to_f64(codes).reshape(codes.shape) * np.repeat(np.repeat(scales, 128, 0), 128, 1)[:256, :384]
    wf = w.astype(np.float64)
    for i in range(2):
        for j in range(3):
            blk = np.abs(wf[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128])
            k = np.unravel_index(np.argmax(blk), blk.shape)
            assert codes[i * 128 + k[0], j * 128 + k[1]] & 0x7F == 0x7E      # the block maximum -> 448
    # relative error of a 3-bit mantissa (half an ulp), absolute near zero (half the subnormal step)
    bound = np.maximum(np.abs(wf) * 2.0 ** -4, 2.0 ** -10 * np.repeat(np.repeat(scales, 128, 0), 128, 1)[:256, :384])
    assert np.all(np.abs(deq - wf) <= bound * 1.0000001)


def test_fp8_all_zero_block_gets_scale_one():
    """Reading of the quantization rule: an all-zero 128 x 128 block has scale
    1 (not 0, which would divide by zero) and zero codes, signs kept."""
    w = (np.random.default_rng(9).standard_normal((128, 256)) * 0.02).astype(np.float16)
    w[:, :128] = 0
    w[5, 7] = -0.0
    codes, scales = oracle.quantize_fp8(w)
    assert scales[0, 0] == F32(1.0) and scales[0, 1] != F32(1.0)
    expect = np.zeros((128, 128), np.uint8)
    expect[5, 7] = 0x80
    assert np.array_equal(codes[:, :128], expect)


def test_nvfp4_quantizer_closed_forms():
    w = np.zeros((4, 64), np.float16)
    w[1, 5] = -3.0                       # the tensor maximum
    w[2, 16:32] = 0.75                   # a constant block
    codes, scales, g = oracle.quantize_nvfp4(w)
    assert g == F32(np.float32(3.0) / F32(2688.0))
    assert scales[1, 0] == 0x7E and scales[0, 0] == 0 and scales[3, 3] == 0
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(4, 64)
    assert nib[1, 5] == 0xF                                   # -6
    assert np.all(nib[0] == 0) and np.all(nib[3] == 0)        # zero blocks: zero codes, zero scales
    assert np.all(nib[2, 16:32] == 7)                         # block max -> +6 at its own scale
    w2 = -np.zeros((1, 16), np.float16)
    c2, s2, g2 = oracle.quantize_nvfp4(w2)
    assert g2 == 1.0 and s2[0, 0] == 0 and np.all(c2 == 0x88)  # signed zeros


def test_nvfp4_quantizer_error_bound():
    w = np.random.default_rng(4).standard_normal((96, 256)).astype(np.float16)
    codes, scales, g = oracle.quantize_nvfp4(w)
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(96, 256).astype(int)
    S = oracle.e4m3_to_f64(scales).reshape(scales.shape)
    deq = oracle.e2m1_to_f64(nib).reshape(nib.shape) * np.repeat(S, 16, 1) * float(g)
    wf = w.astype(np.float64)
    b = np.repeat(np.abs(wf).reshape(96, 16, 16).max(axis=2), 16, 1)
    # the block scale is within 1/16 of b/6 (4-bit mantissa) and an E2M1 step is at most 2 units:
    # every element lands within one code step (2 * S * g) of its value, and within 1/3 of the block max
    assert np.all(np.abs(deq - wf) <= np.repeat(S, 16, 1) * float(g) * 1.0 + 1e-12)
    assert np.all(np.abs(deq - wf) <= b / 3 + 1e-12)


def test_nvfp4_rows_with_the_tensor_maximum_match_the_whole_tensor():
    """Quantizing a subset of rows, given the whole tensor's maximum, gives those
    rows of the whole tensor's result (what the full-size GPU test relies on)."""
    w = (np.random.default_rng(8).standard_normal((64, 256)) * 0.02).astype(np.float16)
    w[7, 3] = -0.5
    codes, scales, g = oracle.quantize_nvfp4(w)
    rows = np.array([0, 7, 40, 63])
    c2, s2, g2 = oracle.quantize_nvfp4(w[rows], amax=np.max(np.abs(w.astype(F32))))
    assert g2 == g
    assert np.array_equal(c2, codes[rows]) and np.array_equal(s2, scales[rows])
    c3, s3, g3 = oracle.quantize_nvfp4(w[rows])            # without it: the subset's own maximum
    assert g3 == g                                          # row 7 holds the maximum here
    c4, _, g4 = oracle.quantize_nvfp4(w[[0, 40]])
    assert g4 != g
