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


# ------------------------------------------------------------------ bfloat16

def bf16_device(a: np.ndarray) -> torch.Tensor:
    """float32 values on the device as bfloat16 (rounded to nearest even on the host)."""
    import normgen
    return torch.from_numpy(normgen.bf16_bits(a).view(np.int16)).to(dev()).view(torch.bfloat16)


def bf16_values(t: torch.Tensor) -> np.ndarray:
    """float32 values of a bfloat16 device tensor (exact)."""
    import normgen
    return normgen.bf16_to_f32(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))


def assert_bf16_parity(got, want, what):
    """|y - y_ref| <= 2^-8 |y_ref| + 1e-4 (1 + |y_ref|) elementwise: the bfloat16 rounding of the
    result plus the fp32 tolerance."""
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    want = np.asarray(want, dtype=np.float64).reshape(-1)
    bound = 2.0**-8 * np.abs(want) + TOL * (1.0 + np.abs(want))
    err = np.abs(got - want)
    bad = ~(err <= bound)
    if bad.any():
        k = int(np.argmax(np.where(bad, err - bound, -np.inf)))
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of bound, worst at {k}: "
                             f"got {got[k]}, want {want[k]}")
