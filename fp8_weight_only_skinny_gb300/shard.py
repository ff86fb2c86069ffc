"""Tensor-parallel shards of a compressed weight, cut on block boundaries.

The pages run the 27B decoder 4-way tensor parallel and quote their kernel
figures "at the actual per-rank shapes" (page "NVFP4 在 Volta 上！", the kernel
table): qkv, gate_up and the lm_head are split over their output features N
(column-parallel), o_proj and down over their input features K
(row-parallel), and each rank reads only its own shard.  A rank's shard is an
ordinary contiguous weight of shape (N / world, K) or (N, K / world) that the
library's calls take as they are; this module cuts it from the full weight.

Cuts must fall on the formats' block boundaries so that every scale belongs
to exactly one shard:
  * NVFP4: one E4M3 scale per 16 consecutive k; a K shard must also keep
    K / world a multiple of 256 (the library's rule for NVFP4 calls).  N may be
    cut anywhere (scales are per row).
  * FP8: one FP32 scale per 128 x 128 block; both cuts must be multiples of 128.
A column-parallel rank computes its rows of y exactly as the full call does
(the same K, so the same per-row summation order): the ranks' outputs
concatenate to the full result bitwise.  A row-parallel rank computes a
partial sum over its K range; the ranks' outputs add up (an all-reduce in a
real deployment) to the full result within the accuracy bound.

Host-side slicing only (PyTorch views, copied to contiguous memory); no
arithmetic of the method happens here.
"""
from __future__ import annotations

AXES = ("n", "k")


def _contig(a):
    """Contiguous copy of a slice of a torch tensor or a numpy array."""
    if hasattr(a, "contiguous"):
        return a.contiguous()
    import numpy as np

    return np.ascontiguousarray(a)


def _range(total: int, rank: int, world: int, align: int, what: str):
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} out of range for world {world}")
    if total % world:
        raise ValueError(f"{what} = {total} does not split into {world} equal shards")
    part = total // world
    if part % align:
        raise ValueError(f"{what} / world = {part} is not a multiple of {align}")
    return rank * part, (rank + 1) * part


def shard_nvfp4(codes, scales, axis: str, rank: int, world: int):
    """Rank `rank` of `world` of an NVFP4 weight (codes u8 [N][K/2], scales u8
    [N][K/16]) cut along `axis` ("n" or "k").  Returns contiguous (codes, scales);
    the tensor scale is shared by every shard."""
    N, K = codes.shape[0], codes.shape[1] * 2
    if tuple(scales.shape) != (N, K // 16):
        raise ValueError("scales must be [N][K/16]")
    if axis == "n":
        n0, n1 = _range(N, rank, world, 1, "N")
        return _contig(codes[n0:n1]), _contig(scales[n0:n1])
    if axis == "k":
        k0, k1 = _range(K, rank, world, 256, "K")
        return _contig(codes[:, k0 // 2:k1 // 2]), _contig(scales[:, k0 // 16:k1 // 16])
    raise ValueError(f"axis must be one of {AXES}")


def shard_fp8(codes, scales, axis: str, rank: int, world: int):
    """Rank `rank` of `world` of an FP8 weight (codes u8 [N][K], scales f32
    [ceil(N/128)][ceil(K/128)]) cut along `axis` ("n" or "k") on 128-blocks.
    Returns contiguous (codes, scales)."""
    N, K = codes.shape
    if tuple(scales.shape) != ((N + 127) // 128, (K + 127) // 128):
        raise ValueError("scales must be [ceil(N/128)][ceil(K/128)]")
    if axis == "n":
        n0, n1 = _range(N, rank, world, 128, "N")
        return _contig(codes[n0:n1]), _contig(scales[n0 // 128:n1 // 128])
    if axis == "k":
        k0, k1 = _range(K, rank, world, 128, "K")
        return _contig(codes[:, k0:k1]), _contig(scales[:, k0 // 128:k1 // 128])
    raise ValueError(f"axis must be one of {AXES}")


def shard_x(x, axis: str, rank: int, world: int):
    """The activations a rank multiplies: all of x for a column-parallel shard,
    its K range (contiguous) for a row-parallel one."""
    if axis == "n":
        return x
    if axis == "k":
        K = x.shape[1]
        k0, k1 = _range(K, rank, world, 1, "K")
        return _contig(x[:, k0:k1])
    raise ValueError(f"axis must be one of {AXES}")
