"""Tensor-parallel shards (fp8_weight_only_skinny_gb300.shard), on the CPU:
the cuts reassemble the full weight, fall on block boundaries, and -- through
the oracle -- column shards reproduce the full output rows exactly while row
shards add up to it."""
import numpy as np
import pytest

import oracle
import synth
from fp8_weight_only_skinny_gb300 import shard


def test_nvfp4_cuts_reassemble_the_weight():
    codes, scales, _ = synth.nvfp4_weights(64, 2048, seed=1)
    for world in (1, 2, 4, 8):
        parts = [shard.shard_nvfp4(codes, scales, "n", r, world) for r in range(world)]
        assert np.array_equal(np.vstack([p[0] for p in parts]), codes)
        assert np.array_equal(np.vstack([p[1] for p in parts]), scales)
        if 2048 // world % 256 == 0:
            parts = [shard.shard_nvfp4(codes, scales, "k", r, world) for r in range(world)]
            assert np.array_equal(np.hstack([p[0] for p in parts]), codes)
            assert np.array_equal(np.hstack([p[1] for p in parts]), scales)
            assert all(p[0].flags["C_CONTIGUOUS"] and p[1].flags["C_CONTIGUOUS"] for p in parts)


def test_fp8_cuts_reassemble_the_weight():
    codes, scales = synth.fp8_weights(512, 1024, seed=2)
    for axis, cat in (("n", np.vstack), ("k", np.hstack)):
        parts = [shard.shard_fp8(codes, scales, axis, r, 4) for r in range(4)]
        assert np.array_equal(cat([p[0] for p in parts]), codes)
        assert np.array_equal(cat([p[1] for p in parts]), scales)


def test_cuts_off_block_boundaries_are_rejected():
    codes, scales, _ = synth.nvfp4_weights(64, 1536, seed=3)
    with pytest.raises(ValueError):
        shard.shard_nvfp4(codes, scales, "k", 0, 4)     # 1536 / 4 = 384 is not a multiple of 256
    with pytest.raises(ValueError):
        shard.shard_nvfp4(codes, scales, "n", 0, 5)     # 64 rows do not split five ways
    c8, s8 = synth.fp8_weights(384, 1024, seed=4)
    with pytest.raises(ValueError):
        shard.shard_fp8(c8, s8, "n", 0, 2)              # 192 rows cut a 128-row scale block
    with pytest.raises(ValueError):
        shard.shard_fp8(c8, s8, "q", 0, 2)
    with pytest.raises(ValueError):
        shard.shard_fp8(c8, s8, "k", 4, 4)


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
def test_column_shards_reproduce_rows_and_row_shards_add_up(fmt):
    M, K, N, world = 3, 2048, 512, 4
    x = synth.x_f16(M, K, seed=5)
    if fmt == "nvfp4":
        codes, scales, g = synth.nvfp4_weights(N, K, seed=6)
        full, _ = oracle.nvfp4_linear(x, codes, scales, g)
        lin = lambda xx, c, s: oracle.nvfp4_linear(xx, c, s, g)[0]
        cut = shard.shard_nvfp4
    else:
        codes, scales = synth.fp8_weights(N, K, seed=6)
        full, _ = oracle.fp8_linear(x, codes, scales)
        lin = lambda xx, c, s: oracle.fp8_linear(xx, c, s)[0]
        cut = shard.shard_fp8
    cols = np.hstack([lin(x, *cut(codes, scales, "n", r, world)) for r in range(world)])
    assert np.array_equal(cols, full)                    # same k order per row: identical
    rows = sum(lin(shard.shard_x(x, "k", r, world), *cut(codes, scales, "k", r, world)) for r in range(world))
    assert np.allclose(rows, full, rtol=1e-12, atol=1e-12)
