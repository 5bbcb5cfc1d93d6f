"""Helpers for the GPU parity tests: guarded device buffers and the parity check."""
from __future__ import annotations

import numpy as np
import torch

TOL = 1e-4  # |y - y_ref| <= TOL * (1 + |y_ref|) elementwise, fp32 against the fp64 oracle
GUARD = 1024  # floats of guard zone before and after every output (4 KB each)
SENTINEL = 0x7FC0DEAD  # a quiet-NaN bit pattern no kernel produces


def dev():
    return torch.device("cuda:0")


class Guarded:
    """A device float32 buffer of n elements with sentinel-filled guard zones.

    ``offset`` shifts the data by that many floats (1 makes it 4- but not 16-byte aligned).
    """

    def __init__(self, n: int, init: np.ndarray | None = None, offset: int = 0):
        self.n = int(n)
        self.lo = GUARD + offset
        self.buf = torch.empty(self.n + 2 * GUARD + offset, dtype=torch.float32, device=dev())
        self.buf.view(torch.int32).fill_(SENTINEL)
        self.t = self.buf[self.lo:self.lo + self.n]
        if init is not None:
            self.t.copy_(torch.from_numpy(np.ascontiguousarray(init, dtype=np.float32)))

    def numpy(self) -> np.ndarray:
        return self.t.cpu().numpy()

    def guards_intact(self) -> bool:
        bits = self.buf.view(torch.int32)
        before = bits[:self.lo]
        after = bits[self.lo + self.n:]
        return bool((before == SENTINEL).all()) and bool((after == SENTINEL).all())


def device(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


def scaled_error(got: np.ndarray, want: np.ndarray) -> float:
    got = np.asarray(got, dtype=np.float64).ravel()
    want = np.asarray(want, dtype=np.float64).ravel()
    assert got.shape == want.shape
    if got.size == 0:
        return 0.0
    if not np.all(np.isfinite(got)):
        return float("inf")
    return float(np.max(np.abs(got - want) / (1.0 + np.abs(want))))


def assert_parity(got, want, what: str, tol: float = TOL):
    err = scaled_error(got, want)
    assert err <= tol, f"{what}: max scaled error {err:.3e} > {tol:.1e}"
    return err
