"""The GPU quantizers' shortcut for the per-weight quotients, checked on the CPU
in IEEE binary32 (numpy float32 divides and multiplies with one rounding to
nearest-even, like the kernels' __fdiv_rn / __fmul_rn).

The codes are defined from q = RN(x / d).  The kernels form p = RN(x * RN(1/d))
and take p's code unless p's bit pattern is within 8 steps of a multiple of
2^19 (E4M3) or 2^21 (E2M1); then they divide.  The rule rests on two facts
pinned here: p is within 6 bit-pattern steps of q, and every rounding boundary
of the code format has a pattern with those low bits zero.  On quotients
crowded around the boundaries (so that p and q often fall on different sides),
every code the rule takes from p must equal q's code, and the rule must also
send to the division the cases where the two codes differ."""
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


E4M3_MASK, E2M1_MASK = (1 << 19) - 1, (1 << 21) - 1


def _accepts(code, p, mask):
    """The kernels' rule: p's code unless p's pattern is within 8 steps of a
    multiple of mask + 1."""
    b = p.view(np.uint32)
    near = ((b + np.uint32(8)) & np.uint32(mask)) < 16
    return ~near, code(p)


def _check(code, q, p, mask, min_rejected_wrong=1):
    ok, c = _accepts(code, p, mask)
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
    _check(e4m3_round, q, p, E4M3_MASK)


def test_nvfp4_codes_from_the_rounded_reciprocal():
    rng = np.random.default_rng(4343)
    n = 400_000
    d = (rng.uniform(1, 2, n) * np.exp2(rng.integers(-40, 8, n))).astype(F32)
    x = _near(_boundaries(oracle.e2m1_to_f64, 8), d, rng, 40)
    q = (x / d).astype(F32)
    p = (x * (F32(1) / d).astype(F32)).astype(F32)
    _check(e2m1_round, q, p, E2M1_MASK)


def test_product_within_six_steps_of_the_quotient():
    """The error bound the 8-step margin rests on: RN(x * RN(1/d)) lies within 3
    units in the last place of x / d's binade from RN(x / d), 6 bit-pattern
    steps at most; over wide ranges of x and d it is never more than 1."""
    rng = np.random.default_rng(4545)
    n = 1_000_000
    d = (rng.uniform(1, 2, n) * np.exp2(rng.integers(-40, 20, n))).astype(F32)
    x = (rng.uniform(1, 2, n) * np.exp2(rng.integers(-20, 16, n))).astype(F32)
    q = (x / d).astype(F32)
    p = (x * (F32(1) / d).astype(F32)).astype(F32)
    dist = np.abs(p.view(np.uint32).astype(np.int64) - q.view(np.uint32).astype(np.int64))
    assert dist.max() <= 1, int(dist.max())
    assert np.count_nonzero(dist) > 0


def test_zero_quotients_are_divided():
    """p = +-0 (x = 0) is a multiple of the grid, so the kernels divide."""
    p = np.array([0.0, -0.0], F32)
    for mask in (E4M3_MASK, E2M1_MASK):
        ok, _ = _accepts(e4m3_round, p, mask)
        assert not ok.any()


def test_every_boundary_is_on_the_grid():
    """Each midpoint between neighbouring E4M3 / E2M1 values (E4M3 subnormals
    included) is a binary32 value whose pattern has the rule's low bits zero."""
    for decode, n, mask in ((oracle.e4m3_to_f64, 0x7F, E4M3_MASK), (oracle.e2m1_to_f64, 8, E2M1_MASK)):
        mids = _boundaries(decode, n)
        m32 = mids.astype(F32)
        assert np.array_equal(m32.astype(np.float64), mids)          # exact in binary32
        assert np.all((m32.view(np.uint32) & np.uint32(mask)) == 0)
        # and the grid is not coarser than needed: a wider mask would miss some
        assert not np.all((m32.view(np.uint32) & np.uint32(2 * mask + 1)) == 0)
