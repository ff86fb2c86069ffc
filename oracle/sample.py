"""CPU oracle for the sampled lm_head pick (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU leg may
import this module; the CUDA path shares nothing with it.

What is computed.  The server the pages describe samples its tokens at a
temperature (page "NVFP4 在 Volta 上！", the "温度 0.6" run) besides the
greedy pick; the pages give no sampler, so this library fixes the usual
temperature / top-k / top-p rule, with the random draw passed in (one
uniform u in [0, 1) per row), for a row of FP32 logits z:

  1. candidates: the top_k largest z, ordered by z descending, ties by the
     lower index;
  2. p_j = exp((z_j - z_0) / T) over the candidates (z_0 the largest);
  3. keep the shortest prefix of the candidates whose summed p reaches
     top_p times the sum over all candidates (at least one);
  4. the pick is the first kept candidate whose running sum of p exceeds
     u times the sum over the kept prefix.
  T <= 0 means the greedy pick (the first candidate).

Here every step after the selection runs in float64 (numpy), so the result
is the exact rule up to the final comparisons; margin() reports how far
those comparisons are from a tie, for tests that compare with an FP32
implementation.

Parity status: pinned (tests/test_oracle_sample.py).
"""
from __future__ import annotations

import numpy as np


def _order(z):
    z = np.asarray(z, dtype=np.float32)
    # descending value, then ascending index (lexsort sorts by the last key first)
    return np.lexsort((np.arange(z.size), -z.astype(np.float64)))


def sample_row(z, u, temperature, top_k, top_p):
    """The pick (token index) of one row of FP32 logits z."""
    order = _order(z)[:top_k]
    if temperature <= 0:
        return int(order[0])
    zz = np.asarray(z, dtype=np.float32)[order].astype(np.float64)
    p = np.exp((zz - zz[0]) / float(np.float32(temperature)))
    cum = np.cumsum(p)
    keep = int(np.searchsorted(cum, float(np.float32(top_p)) * cum[-1], side="left")) + 1
    keep = min(max(keep, 1), order.size)
    target = float(np.float32(u)) * cum[keep - 1]
    j = int(np.searchsorted(cum[:keep], target, side="right"))
    return int(order[min(j, keep - 1)])


def margin(z, u, temperature, top_k, top_p):
    """Relative distance of this row's two decisions (the top-p cut and the
    draw) from a tie: the smaller of |cum_j - threshold| / cum_total over the
    boundaries next to each decision.  Below ~1e-5 an FP32 sum may decide
    the other way."""
    order = _order(z)[:top_k]
    if temperature <= 0:
        return np.inf
    zz = np.asarray(z, dtype=np.float32)[order].astype(np.float64)
    p = np.exp((zz - zz[0]) / float(np.float32(temperature)))
    cum = np.cumsum(p)
    tot = cum[-1]
    thr = float(np.float32(top_p)) * tot
    keep = min(max(int(np.searchsorted(cum, thr, side="left")) + 1, 1), order.size)
    target = float(np.float32(u)) * cum[keep - 1]
    # the cut moves only if the threshold crosses the sum just before it, or
    # (when there is a next candidate) the sum at it
    d = np.inf
    if keep >= 2:
        d = min(d, thr - cum[keep - 2])
    if keep < order.size:
        d = min(d, cum[keep - 1] - thr)
    d2 = np.min(np.abs(cum[:keep] - target))
    return float(min(d, d2) / tot)


def sample(logits, u, temperature, top_k, top_p):
    """Picks for every row of logits [M][N] with uniforms u [M]."""
    logits = np.asarray(logits, dtype=np.float32)
    return np.array([sample_row(logits[m], u[m], temperature, top_k, top_p) for m in range(logits.shape[0])],
                    dtype=np.int64)
