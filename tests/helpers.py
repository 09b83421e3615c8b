"""Helpers of the GPU parity tests: guarded output buffers and the fp64 oracle run
over heads on every host core.

Guarded outputs
    Every output (and workspace) a parity test hands to the library is a view
    into a larger device buffer: 256 canary bytes in front, the output itself
    (also filled with the canary, so that an element the kernel forgets to
    write shows up as a wrong value), then 4096 canary bytes behind.  After the
    call the test checks that both guard regions still hold the canary, so a
    write before the start or past the end of an output fails the test.  The
    front guard keeps the output 256-byte aligned.

Oracle over heads
    The oracle computes one (batch, head) slice at a time; the full-size checks
    hand the slices to a thread pool (numpy's matrix products and element-wise
    passes release the interpreter lock; the test session limits BLAS to one
    thread per call, see ``conftest.py``).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GUARD_FRONT = 256
GUARD_TAIL = 4096
CANARY = 0xA5


class Guarded:
    """A device output of ``shape`` / ``dtype`` with canary bytes on both sides."""

    def __init__(self, shape, dtype, device):
        import torch
        self.shape = tuple(int(x) for x in shape)
        esize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = math.prod(self.shape) * esize
        self.buf = torch.full((GUARD_FRONT + self.nbytes + GUARD_TAIL,), CANARY, dtype=torch.uint8, device=device)
        self.t = self.buf[GUARD_FRONT:GUARD_FRONT + self.nbytes].view(dtype).view(self.shape)

    def check(self, name="output"):
        """Both guard regions must still hold the canary (call after the stream is synchronised)."""
        front = self.buf[:GUARD_FRONT]
        tail = self.buf[GUARD_FRONT + self.nbytes:]
        bad_front = int((front != CANARY).sum())
        bad_tail = int((tail != CANARY).sum())
        assert bad_front == 0 and bad_tail == 0, (
            f"{name}: {bad_front} byte(s) written before the start and {bad_tail} past the end")


def guarded(shape, dtype, device):
    return Guarded(shape, dtype, device)


def check_guards(*gs):
    import torch
    torch.cuda.synchronize()
    for i, g in enumerate(gs):
        if g is not None:
            g.check(f"buffer {i} {tuple(g.shape)}")


def host_threads():
    return max(1, len(os.sched_getaffinity(0)))


def parallel_map(fn, items, threads=None):
    """``[fn(x) for x in items]`` on a thread pool of every host core."""
    with ThreadPoolExecutor(threads or host_threads()) as ex:
        return list(ex.map(fn, items))


def compare_rows(o, lse, O, L, lse_relative=True):
    """(max-abs O error, LSE error, finiteness agrees) of a GPU slice against the oracle's.

    LSE error is ``|dLSE| / max(1, |LSE|)`` (relative) or ``|dLSE|``; -inf entries
    must agree exactly and are excluded from the error.
    """
    o = np.asarray(o, dtype=np.float64).reshape(O.shape)
    l = np.asarray(lse, dtype=np.float64).reshape(L.shape)
    finite_out = bool(np.isfinite(o).all())
    err_o = float(np.abs(o - O).max()) if O.size else 0.0
    fin = np.isfinite(L)
    fin_ok = finite_out and np.array_equal(np.isfinite(l), fin) and bool(np.all(l[~fin] == -np.inf))
    err_l = 0.0
    if fin.any() and fin_ok:
        d = np.abs(l[fin] - L[fin])
        if lse_relative:
            d = d / np.maximum(1.0, np.abs(L[fin]))
        err_l = float(d.max())
    return err_o, err_l, fin_ok
