"""The GPU quantizers' shortcut for the per-weight quotients, checked on the CPU
in IEEE binary32 (numpy float32 divides and multiplies with one rounding to
nearest-even, like the kernels' __fdiv_rn / __fmul_rn).

The codes are defined from q = RN(x / d).  The kernels form p = RN(x * RN(1/d))
and take p's code when the bit patterns `steps` below and above p round to the
same code; otherwise they divide.  Here, on quotients crowded around the
E4M3 / E2M1 rounding boundaries (so that p and q often fall on different sides),
every accepted code must equal q's code, and the test must also reject the cases
where the two codes differ (E4M3 for fp8_quantize, E2M1 for nvfp4_quantize, 8
steps for both)."""
import numpy as np

import oracle
from oracle.quant import e2m1_round, e4m3_round

F32 = np.float32


def _boundaries(decode, ncodes):
    vals = np.unique(decode(np.arange(ncodes)))
    vals = vals[np.isfinite(vals) & (vals >= 0)]
    return (vals[:-1] + vals[1:]) / 2          # midpoints between neighbouring values


def _near(mids, d, rng, spread):
    """x (float32) with x / d within about `spread` units in the last place of a midpoint."""
    m = mids[rng.integers(0, mids.size, d.size)]
    k = rng.integers(-spread, spread + 1, d.size)
    sign = rng.choice([-1.0, 1.0], d.size)
    return (sign * m * d.astype(np.float64) * (1 + k * 2.0 ** -24)).astype(F32)


def _steps(p, n):
    b = p.view(np.uint32)
    lo = (b - np.uint32(n)).astype(np.uint32).view(F32)
    hi = (b + np.uint32(n)).astype(np.uint32).view(F32)
    return lo, hi


def _accepts(code, p, n):
    lo, hi = _steps(p, n)
    with np.errstate(invalid="ignore"):
        c, cl, ch = code(p), code(lo), code(hi)
    nan = np.isnan(lo) | np.isnan(hi)          # the kernels' conversion gives a NaN code there
    return (c == cl) & (c == ch) & ~nan, c


def _check(code, q, p, n, min_rejected_wrong=1):
    ok, c = _accepts(code, p, n)
    cq = code(q)
    assert ok.mean() > 0.4, ok.mean()                       # the shortcut is taken most of the time
    assert np.array_equal(c[ok], cq[ok]), int(np.sum(c[ok] != cq[ok]))
    wrong = (c != cq) & ~ok
    assert wrong.sum() >= min_rejected_wrong                # cases where p alone would have been wrong


def test_fp8_codes_from_the_rounded_reciprocal():
    rng = np.random.default_rng(4242)
    n = 400_000
    d = (rng.uniform(1, 2, n) * np.exp2(rng.integers(-12, 4, n))).astype(F32)
    x = _near(_boundaries(oracle.e4m3_to_f64, 0x7F), d, rng, 40)
    q = (x / d).astype(F32)
    r = (F32(1) / d).astype(F32)
    p = (x * r).astype(F32)
    _check(e4m3_round, q, p, 8)


def test_nvfp4_codes_from_the_rounded_reciprocal():
    rng = np.random.default_rng(4343)
    n = 400_000
    d = (rng.uniform(1, 2, n) * np.exp2(rng.integers(-40, 8, n))).astype(F32)
    x = _near(_boundaries(oracle.e2m1_to_f64, 8), d, rng, 40)
    q = (x / d).astype(F32)
    p = (x * (F32(1) / d).astype(F32)).astype(F32)
    _check(e2m1_round, q, p, 8)


def test_product_within_three_steps_of_the_quotient():
    """The error bound the 8-step test rests on: RN(x * RN(1/d)) lies within 3
    bit-pattern steps of RN(x / d), over wide ranges of x and d."""
    rng = np.random.default_rng(4545)
    n = 1_000_000
    d = (rng.uniform(1, 2, n) * np.exp2(rng.integers(-40, 20, n))).astype(F32)
    x = (rng.uniform(1, 2, n) * np.exp2(rng.integers(-20, 16, n))).astype(F32)
    q = (x / d).astype(F32)
    p = (x * (F32(1) / d).astype(F32)).astype(F32)
    dist = np.abs(p.view(np.uint32).astype(np.int64) - q.view(np.uint32).astype(np.int64))
    assert dist.max() <= 3, int(dist.max())
    assert np.count_nonzero(dist) > 0


def test_zero_quotients_are_divided():
    """p = +-0 (x = 0): 8 steps below is a NaN pattern, so the kernels divide."""
    p = np.array([0.0, -0.0], F32)
    ok, _ = _accepts(e4m3_round, p, 8)
    assert not ok.any()
