"""Helpers shared by the GPU tests: device placement, guarded output buffers
and oracle comparison."""
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


CANARY = 0xA5
GUARD_BYTES = 4096


class Guarded:
    """An output tensor placed between two guard bands of canary bytes.

    compute-sanitizer is not available where the GPU tests run, so an
    out-of-bounds store past the end (or before the start) of an output would
    otherwise go unnoticed whenever the neighbouring memory is unused.  The
    tensor `t` sits inside one larger allocation; the GUARD_BYTES before and
    after it hold CANARY and check() asserts that they still do.  The tensor
    itself starts out filled with `fill` (NaN by default, so an output element
    the kernel never writes fails the comparison with the oracle)."""

    def __init__(self, shape, dtype, fill=float("nan")):
        import torch

        self.shape = tuple(int(s) for s in shape)
        n = int(np.prod(self.shape)) if self.shape else 1
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((2 * GUARD_BYTES + self.nbytes,), CANARY, dtype=torch.uint8, device="cuda:0")
        self.t = self.buf[GUARD_BYTES:GUARD_BYTES + self.nbytes].view(dtype).view(self.shape)
        if fill is not None:
            self.t.fill_(fill)

    def check(self, what=""):
        import torch

        torch.cuda.synchronize()
        pre = self.buf[:GUARD_BYTES].cpu().numpy()
        post = self.buf[GUARD_BYTES + self.nbytes:].cpu().numpy()
        for name, band in (("before", pre), ("after", post)):
            bad = np.flatnonzero(band != CANARY)
            assert bad.size == 0, (f"{what}: {bad.size} guard bytes {name} the output were overwritten "
                                   f"(first at offset {int(bad[0])} of the band)")

    def host(self, what=""):
        """The tensor's contents (as host()), after checking both guard bands."""
        a = host(self.t)
        self.check(what)
        return a


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


def argmax_ok(am, y_ref, l1, logits_gpu=None):
    """The greedy pick against the oracle: where the oracle's top-2 gap exceeds
    the two tolerances the index must be the oracle's (lowest-index) argmax
    exactly; otherwise any index whose oracle logit is within tolerance of the
    maximum is accepted.  With logits_gpu, the pick must also be the
    lowest-index maximum of the same call's FP32 logits, bitwise.
    Returns the number of rows decided by the gap rule."""
    M = y_ref.shape[0]
    tol = oracle.tolerance(l1)
    strict = 0
    for m in range(M):
        if logits_gpu is not None:
            assert am[m] == int(np.argmax(logits_gpu[m])), m
        a = int(oracle.argmax_rows(y_ref[m:m + 1])[0])
        order = np.argsort(-y_ref[m], kind="stable")
        b = int(order[1]) if order[0] == a else int(order[0])
        if y_ref[m, a] - y_ref[m, b] > tol[m, a] + tol[m, b]:
            assert am[m] == a, (m, int(am[m]), a)
            strict += 1
        else:
            i = int(am[m])
            assert y_ref[m, i] >= y_ref[m, a] - tol[m, a] - tol[m, i], (m, i, a)
    return strict
