"""Pins of the sampling oracle (oracle/sample.py) on the CPU: a stratified
sweep of the uniform draw reproduces the renormalised top-k / top-p
probabilities written out by hand, and the degenerate settings reduce to the
greedy pick."""
import math

import numpy as np
import pytest

import oracle


def _expected(z, T, k, p):
    """The sampling distribution, written out directly: candidates sorted by
    (value desc, index asc), softmax at temperature T, top-p prefix, renormalised."""
    cand = sorted(range(len(z)), key=lambda i: (-float(z[i]), i))[:k]
    w = [math.exp((float(z[i]) - float(z[cand[0]])) / T) for i in cand]
    tot, run, kept = sum(w), 0.0, []
    for i, wi in zip(cand, w):
        kept.append((i, wi))
        run += wi
        if run >= p * tot:
            break
    s = sum(wi for _, wi in kept)
    return {i: wi / s for i, wi in kept}


@pytest.mark.parametrize("T,k,p", [(1.0, 10, 1.0), (0.6, 10, 0.9), (2.0, 4, 0.5), (0.3, 20, 0.95)])
def test_stratified_draws_reproduce_the_distribution(T, k, p):
    z = np.random.default_rng(7).standard_normal(40).astype(np.float32)
    z[3] = z[5] = np.float32(2.5)                                  # a tie among the top values
    n = 20000
    picks = [oracle.sample_row(z, (i + 0.5) / n, T, k, p) for i in range(n)]
    want = _expected(z, T, k, p)
    counts = {i: picks.count(i) / n for i in set(picks)}
    assert set(counts) == set(want)
    for i, q in want.items():
        assert abs(counts[i] - q) <= 2.0 / n, (i, counts[i], q)


def test_degenerate_settings_give_the_greedy_pick():
    z = np.array([0.5, 3.0, 1.0, 3.0, -2.0], np.float32)
    for u in (0.0, 0.3, 0.999):
        assert oracle.sample_row(z, u, 0.0, 5, 1.0) == 1           # T <= 0: greedy, ties to the lower index
        assert oracle.sample_row(z, u, 1.0, 1, 1.0) == 1           # top_k = 1
        assert oracle.sample_row(z, u, 1.0, 5, 1e-9) == 1          # top_p ~ 0 keeps one token
    assert oracle.sample_row(z, 0.9999, 1.0, 2, 1.0) == 3          # the tied runner-up
    assert oracle.sample_row(z, 0.0, 1e9, 5, 1.0) == 1             # u = 0 always gives the first


def test_margin_flags_near_ties():
    z = np.array([0.0, 0.0], np.float32)                          # two equal tokens: cum = 1, 2
    assert oracle.sample_margin(z, 0.5, 1.0, 2, 1.0) == 0.0        # u * 2 = 1 sits on the boundary
    assert oracle.sample_margin(z, 0.25, 1.0, 2, 1.0) == pytest.approx(0.25)
