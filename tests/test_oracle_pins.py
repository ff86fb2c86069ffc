"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties one part of ``oracle/`` to something independent of it: a value
table from a format specification (tests/golden), a library conversion routine
(numpy float16, torch float8_e4m3fn), a hand-worked example, a closed form, or
an invariant of the exact product.  Together they catch a dropped term, a sign
error, a wrong index (nibble order, block-scale index, row/column swap) or a
transposed operand anywhere in the oracle.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth


def _read_table(path):
    out = {}
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        a, b = line.split()
        out[int(a, 16)] = float(b)
    return out


def _kv(path):
    out = {}
    for line in open(path):
        line = line.split("#")[0].strip()
        if line:
            k, *v = line.split()
            out[k] = v
    return out


@pytest.fixture(scope="module")
def e2m1_table(golden_dir):
    t = _read_table(os.path.join(golden_dir, "e2m1_values.txt"))
    assert sorted(t) == list(range(16))
    return np.array([t[i] for i in range(16)], np.float64)


def _e4m3_lib(codes):
    """E4M3 decode by the library routine (torch float8_e4m3fn -> float32)."""
    c = torch.from_numpy(np.ascontiguousarray(np.asarray(codes, np.uint8)))
    return c.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def _same(a, b):
    """Bitwise-equal values (signed zeros told apart); NaN matches any NaN."""
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    na, nb = np.isnan(a), np.isnan(b)
    if not np.array_equal(na, nb):
        return False
    a, b = a[~na], b[~nb]
    return np.array_equal(a, b) and np.array_equal(np.signbit(a), np.signbit(b))


# ---------------------------------------------------------------- decoders ---

def test_f16_all_codes_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    assert _same(oracle.f16_to_f64(bits), ref)


def test_e2m1_all_codes_match_spec_table(e2m1_table):
    got = oracle.e2m1_to_f64(np.arange(16))
    assert _same(got, e2m1_table)


def test_e4m3_all_codes_match_library():
    codes = np.arange(256, dtype=np.uint32).astype(np.uint8)
    assert _same(oracle.e4m3_to_f64(codes), _e4m3_lib(codes))


def test_e4m3_landmarks_match_spec(golden_dir):
    pts = _read_table(os.path.join(golden_dir, "e4m3_points.txt"))
    codes = np.array(sorted(pts), np.uint8)
    assert _same(oracle.e4m3_to_f64(codes), np.array([pts[c] for c in sorted(pts)]))


# ------------------------------------------------------- hand-worked cases ---

def test_tiny_nvfp4_hand_example(golden_dir):
    g = _kv(os.path.join(golden_dir, "tiny_nvfp4.txt"))
    x = np.array([[float(v) for v in g["x"]]], np.float16)
    codes = np.array([[int(v, 16) for v in g["codes"]]], np.uint8)
    scales = np.array([[int(v, 16) for v in g["scales"]]], np.uint8)
    y, l1 = oracle.nvfp4_linear(x, codes, scales, float(g["gscale"][0]))
    assert y[0, 0] == float(g["y"][0])
    assert l1[0, 0] == float(g["l1"][0])


def test_tiny_fp8_hand_example(golden_dir):
    g = _kv(os.path.join(golden_dir, "tiny_fp8.txt"))
    K, N = int(g["K"][0]), int(g["N"][0])
    codes = np.full((N, K), int(g["code"][0], 16), np.uint8)
    scales = np.array([float(v) for v in g["scales"]], np.float32).reshape(2, 2)
    x = np.ones((1, K), np.float16)
    y, _ = oracle.fp8_linear(x, codes, scales)
    assert np.all(y[0, :128] == float(g["y_rows_0_127"][0]))
    assert np.all(y[0, 128:] == float(g["y_rows_128_129"][0]))


# ---------------------------------------------------------------- identity ---

def test_nvfp4_identity_returns_x_bitwise():
    K = N = 512
    x = synth.x_f16(3, K, seed=11)
    nib = np.zeros((N, K), np.uint8)
    nib[np.arange(N), np.arange(K)] = 0x2                      # E2M1 1.0
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    scales = np.full((N, K // 16), 0x38, np.uint8)               # E4M3 1.0
    y, _ = oracle.nvfp4_linear(x, codes, scales, 1.0)
    assert np.array_equal(y, x.astype(np.float64))


def test_fp8_identity_returns_x_bitwise():
    K = N = 512
    x = synth.x_f16(2, K, seed=12)
    codes = np.zeros((N, K), np.uint8)
    codes[np.arange(N), np.arange(K)] = 0x38
    scales = np.ones((4, 4), np.float32)
    y, _ = oracle.fp8_linear(x, codes, scales)
    assert np.array_equal(y, x.astype(np.float64))


# ----------------------------------------------------------------- one-hot ---

@pytest.mark.parametrize("k0", [0, 1, 14, 15, 16, 17, 31, 127, 128, 129, 255])
@pytest.mark.parametrize("n0", [0, 1, 5, 19])
def test_nvfp4_one_hot_selects_the_right_code_and_scale(e2m1_table, k0, n0):
    M, N, K = 2, 20, 256
    x = synth.x_f16(M, K, seed=100 + k0)
    for c in (0x1, 0x7, 0x9, 0xF):
        nib = np.zeros((N, K), np.uint8)
        nib[n0, k0] = c
        codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
        # every block scale distinct, so a wrong block index changes the value
        scales = (0x20 + (np.arange(N * (K // 16)) % 48)).astype(np.uint8).reshape(N, K // 16)
        g = 0.75
        y, _ = oracle.nvfp4_linear(x, codes, scales, g)
        s = _e4m3_lib([scales[n0, k0 // 16]])[0]
        want = x[:, k0].astype(np.float64) * e2m1_table[c] * s * g
        assert np.array_equal(y[:, n0], want)
        others = np.delete(y, n0, axis=1)
        assert np.all(others == 0)


@pytest.mark.parametrize("k0,n0", [(0, 0), (127, 127), (128, 128), (129, 5), (200, 131), (255, 129)])
def test_fp8_one_hot_selects_the_right_block_scale(k0, n0):
    M, N, K = 3, 140, 256
    x = synth.x_f16(M, K, seed=7)
    codes = np.zeros((N, K), np.uint8)
    codes[n0, k0] = 0x3A                                            # E4M3 1.25
    scales = np.array([[0.5, 2.0], [4.0, 0.25]], np.float32)
    y, _ = oracle.fp8_linear(x, codes, scales)
    want = x[:, k0].astype(np.float64) * 1.25 * float(scales[n0 // 128, k0 // 128])
    assert np.array_equal(y[:, n0], want)
    assert np.all(np.delete(y, n0, axis=1) == 0)


# ------------------------------------------------------------- closed form ---

@pytest.mark.parametrize("c,s", [(0x2, 0x38), (0x5, 0x18), (0xB, 0x58), (0x7, 0x41)])
def test_nvfp4_constant_weights_closed_form(e2m1_table, c, s):
    M, N, K = 2, 3, 512
    x = synth.x_f16(M, K, seed=c * 256 + s)
    codes = np.full((N, K // 2), c | (c << 4), np.uint8)
    scales = np.full((N, K // 16), s, np.uint8)
    g = float(np.float32(0.01))
    y, _ = oracle.nvfp4_linear(x, codes, scales, g)
    w = e2m1_table[c] * _e4m3_lib([s])[0] * g
    for m in range(M):
        want = math.fsum(float(v) * w for v in x[m])
        assert y[m, 0] == pytest.approx(want, rel=1e-14, abs=1e-300)
        assert np.all(y[m] == y[m, 0])


# -------------------------------------------- library-routine special case ---

def _nvfp4_dense_via_table(codes, scales, g, e2m1_table):
    N = codes.shape[0]
    nib = np.empty((N, codes.shape[1] * 2), np.uint8)
    nib[:, 0::2] = codes & 0xF
    nib[:, 1::2] = codes >> 4
    s = _e4m3_lib(scales.ravel()).reshape(scales.shape)
    return e2m1_table[nib] * np.repeat(s, 16, axis=1) * g


def test_nvfp4_matches_table_decode_and_numpy_matmul(e2m1_table):
    M, N, K = 4, 96, 1024
    x = synth.x_f16(M, K, seed=3)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=3)
    y, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    W = _nvfp4_dense_via_table(codes, scales, float(g), e2m1_table)
    xf = x.astype(np.float64)
    ref = xf @ W.T
    assert np.allclose(y, ref, rtol=0, atol=1e-12 * np.abs(xf) @ np.abs(W).T + 1e-300)
    assert np.allclose(l1, np.abs(xf) @ np.abs(W).T, rtol=1e-13, atol=0)


def test_fp8_matches_library_decode_and_numpy_matmul():
    M, N, K = 3, 200, 384
    x = synth.x_f16(M, K, seed=4)
    codes, scales = synth.fp8_weights(N, K, seed=4)
    y, l1 = oracle.fp8_linear(x, codes, scales)
    W = _e4m3_lib(codes.ravel()).reshape(N, K) * np.repeat(
        np.repeat(scales.astype(np.float64), 128, 0), 128, 1)[:N, :K]
    xf = x.astype(np.float64)
    assert np.allclose(y, xf @ W.T, rtol=0, atol=1e-12 * np.abs(xf) @ np.abs(W).T + 1e-300)
    assert np.allclose(l1, np.abs(xf) @ np.abs(W).T, rtol=1e-13, atol=0)


def test_fp8_generator_roundtrip_is_close_to_source():
    """Generated FP8 weights decode to within E4M3 rounding of N(0,0.02) samples."""
    N, K = 130, 300
    g = synth.rng(9, "fp8", N, K, 0)
    w = g.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    codes, scales = synth.fp8_quantize(w)
    W = _e4m3_lib(codes.ravel()).reshape(N, K) * np.repeat(
        np.repeat(scales.astype(np.float64), 128, 0), 128, 1)[:N, :K]
    blockmax = np.repeat(np.repeat(scales.astype(np.float64) * 448, 128, 0), 128, 1)[:N, :K]
    # E4M3 has 3 mantissa bits: relative error <= 2^-4 for normals, absolute
    # error <= 2^-10 * block scale for subnormals.
    err = np.abs(W - w)
    assert np.all(err <= np.maximum(np.abs(w) * 2.0 ** -4, blockmax / 448 * 2.0 ** -10) * 1.0001)


# --------------------------------------------------------------- invariants ---

def test_power_of_two_scaling_is_exact():
    M, N, K = 2, 16, 512
    x = synth.x_f16(M, K, seed=5)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=5)
    y, _ = oracle.nvfp4_linear(x, codes, scales, g)
    y4, _ = oracle.nvfp4_linear((x.astype(np.float32) * 4).astype(np.float16), codes, scales, g)
    assert np.array_equal(y4, 4 * y)
    y2, _ = oracle.nvfp4_linear(x, codes, scales, np.float32(2 * g))
    assert np.array_equal(y2, 2 * y)
    c8, s8 = synth.fp8_weights(N, K, seed=5)
    f, _ = oracle.fp8_linear(x, c8, s8)
    f8, _ = oracle.fp8_linear((x.astype(np.float32) / 8).astype(np.float16), c8, s8)
    assert np.array_equal(f8, f / 8)


def test_additivity_over_disjoint_k_support():
    M, N, K = 2, 24, 512
    x = synth.x_f16(M, K, seed=6)
    x1 = x.copy(); x1[:, K // 2:] = 0
    x2 = x.copy(); x2[:, :K // 2] = 0
    codes, scales, g = synth.nvfp4_weights(N, K, seed=6)
    y, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    ya, _ = oracle.nvfp4_linear(x1, codes, scales, g)
    yb, _ = oracle.nvfp4_linear(x2, codes, scales, g)
    assert np.all(np.abs(y - (ya + yb)) <= 1e-12 * l1)
    # and sign: negating x negates y exactly
    yn, _ = oracle.nvfp4_linear(-x, codes, scales, g)
    assert np.array_equal(yn, -y)


def test_rows_are_independent():
    N, K = 40, 256
    x = synth.x_f16(8, K, seed=8)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=8)
    y, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    c8, s8 = synth.fp8_weights(N, K, seed=8)
    f, _ = oracle.fp8_linear(x, c8, s8)
    for m in range(8):
        ym, lm = oracle.nvfp4_linear(x[m:m + 1], codes, scales, g)
        assert np.array_equal(ym[0], y[m]) and np.array_equal(lm[0], l1[m])
        fm, _ = oracle.fp8_linear(x[m:m + 1], c8, s8)
        assert np.array_equal(fm[0], f[m])


def test_column_subset_equals_full_columns():
    N, K = 50, 256
    x = synth.x_f16(3, K, seed=9)
    codes, scales, g = synth.nvfp4_weights(N, K, seed=9)
    y, l1 = oracle.nvfp4_linear(x, codes, scales, g)
    cols = [49, 0, 17, 17, 3]
    ys, ls = oracle.nvfp4_linear(x, codes, scales, g, cols=cols)
    assert np.array_equal(ys, y[:, cols]) and np.array_equal(ls, l1[:, cols])


# ------------------------------------------------------------------ argmax ---

def test_argmax_ties_go_to_lowest_index_and_match_numpy():
    y = np.array([[1.0, 3.0, 3.0, -1.0],
                  [-2.0, -2.0, -5.0, -2.0],
                  [0.0, -0.0, 0.0, 0.0],
                  [np.nan, 2.0, np.nan, 2.0]])
    assert list(oracle.argmax_rows(y)) == [1, 0, 0, 1]
    r = np.random.default_rng(0).integers(-3, 4, size=(16, 257)).astype(np.float64)
    assert np.array_equal(oracle.argmax_rows(r), np.argmax(r, axis=1))


def test_tolerance_formula():
    assert oracle.tolerance(np.array([3.5]))[0] == pytest.approx(3.5e-3 + 1e-6)
    # one FP16 ulp at 1.0 is 2^-10, at 1000 it is 2^-1, below 2^-14 it is 2^-24
    t = oracle.tolerance(np.zeros(3), f16_out=True, y_ref=np.array([1.0, 1000.0, 1e-6]))
    assert np.allclose(t - 1e-6, [2.0 ** -10, 2.0 ** -1, 2.0 ** -24])


# ---------------------------------------------------------- verify round ---

def _committed_by_enumeration(target, draft):
    """The committed tokens of a greedy speculative round, by direct enumeration:
    the longest prefix of the drafts that the target would have produced itself
    token by token, then the target's own next token."""
    out = []
    for j in range(len(target)):
        out.append(int(target[j]))           # the target's pick at this position is committed
        if j == len(target) - 1 or int(draft[j]) != int(target[j]):
            break                            # a rejected draft ends the round after the target's pick
    return out


def test_verify_matches_enumeration_on_every_tiny_case():
    """Every target and draft sequence over a two-token alphabet for M = 1..5:
    the accepted count and bonus token reproduce the committed sequence."""
    import itertools
    for M in range(1, 6):
        for target in itertools.product((0, 1), repeat=M):
            for draft in itertools.product((0, 1), repeat=M - 1):
                a, bonus = oracle.verify(np.array(target), np.array(draft, dtype=np.int32))
                committed = _committed_by_enumeration(target, draft)
                assert len(committed) == a + 1 and committed[-1] == bonus, (target, draft)
                assert list(draft[:a]) == committed[:-1]


def test_verify_special_cases():
    t = np.array([7, 11, 13, 17, 19, 23, 29, 31])
    assert oracle.verify(t, t[:7].astype(np.int32)) == (7, 31)          # every draft accepted
    assert oracle.verify(t, np.full(7, -1, np.int32)) == (0, 7)         # first draft rejected
    assert oracle.verify(t[:1], np.zeros(0, np.int32)) == (0, 7)       # one row: no drafts
    for L in range(7):                                                  # first mismatch at L
        d = t[:7].astype(np.int32).copy()
        d[L] = 1000
        assert oracle.verify(t, d) == (L, int(t[L]))
