"""Helpers shared by the GPU tests: device placement and oracle comparison."""
import contextlib

import numpy as np

import oracle


def dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda:0")


@contextlib.contextmanager
def variant(sk, name):
    """Run the block with the kernel variant `name` ("auto", "tensor" or "simt")."""
    code = {"auto": sk.VARIANT_AUTO, "tensor": sk.VARIANT_TENSOR, "simt": sk.VARIANT_SIMT}[name]
    prev = sk.set_variant(code)
    try:
        yield
    finally:
        sk.set_variant(prev)


def host(t):
    import torch

    torch.cuda.synchronize()
    a = t.cpu().numpy()
    return a.astype(np.float64) if a.dtype in (np.float16, np.float32) else a


def check(y_gpu, y_ref, l1, f16_out=False, what=""):
    """Element-wise accuracy contract; returns the worst err / tolerance ratio."""
    y_gpu = np.asarray(y_gpu, np.float64)
    tol = oracle.tolerance(l1, f16_out=f16_out, y_ref=y_ref)
    err = np.abs(y_gpu - y_ref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}: "
            f"gpu={y_gpu[tuple(i)]!r} ref={y_ref[tuple(i)]!r} tol={tol[tuple(i)]!r}")
    return float(np.max(err / tol)) if err.size else 0.0
