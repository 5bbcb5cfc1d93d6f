"""Seeded, counter-based synthetic inputs shared by the oracle's tests and the CUDA path.

The generator (``normgen.c``) is SplitMix64 with Box-Muller for normal draws; its
header comment gives the exact stream definition.  Element ``i`` of a tensor
depends only on ``(seed, tensor_id, i)``, so any sub-range can be produced on its
own and the bytes do not depend on the thread count.  Nothing in this module
computes any part of a normalization.

Tensor ids used throughout the repository: 0 = x, 1 = gamma, 2 = beta, and for the
Linear that feeds GroupNorm 3 = its weight W, 4 = its bias.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "normgen.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libnormgen.so")

TENSOR_X = 0
TENSOR_GAMMA = 1
TENSOR_BETA = 2
TENSOR_W = 3
TENSOR_LIN_BIAS = 4

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile normgen.c into ``_build/libnormgen.so`` (plain gcc, no SIMD flags)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(_LIB_DIR, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_LIB_DIR)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            for name in ("normgen_fill_normal", "normgen_fill_uniform"):
                fn = getattr(lib, name)
                fn.restype = ctypes.c_int
                fn.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                               ctypes.c_double, ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
            lib.normgen_splitmix64_output.restype = ctypes.c_uint64
            lib.normgen_splitmix64_output.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.normgen_word.restype = ctypes.c_uint64
            lib.normgen_word.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _target(n: int, out):
    if out is None:
        return np.empty(n, dtype=np.float32)
    if out.dtype != np.float32 or not out.flags["C_CONTIGUOUS"] or out.size != n:
        raise ValueError("out must be a contiguous float32 array of n elements")
    return out.reshape(-1)


def normal(n: int, mean: float = 0.0, std: float = 1.0, *, seed: int = 0, tensor_id: int = 0,
           start: int = 0, threads: int | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """Elements ``start .. start+n-1`` of the N(mean, std^2) stream for (seed, tensor_id), as float32."""
    n = int(n)
    dst = _target(n, out)
    rc = _load().normgen_fill_normal(seed, tensor_id, start, n, float(mean), float(std),
                                     dst.ctypes.data, threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"normgen_fill_normal failed ({rc})")
    return dst if out is None else out


def uniform(n: int, lo: float = 0.0, hi: float = 1.0, *, seed: int = 0, tensor_id: int = 0,
            start: int = 0, threads: int | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """Elements ``start .. start+n-1`` of the U(lo, hi) stream for (seed, tensor_id), as float32."""
    n = int(n)
    dst = _target(n, out)
    rc = _load().normgen_fill_uniform(seed, tensor_id, start, n, float(lo), float(hi),
                                      dst.ctypes.data, threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"normgen_fill_uniform failed ({rc})")
    return dst if out is None else out


def word(seed: int, tensor_id: int, k: int) -> int:
    """The k-th raw 64-bit SplitMix64 word of the (seed, tensor_id) stream."""
    return int(_load().normgen_word(seed, tensor_id, k))


def splitmix64_output(s0: int, k: int) -> int:
    """The k-th output of a plain SplitMix64 generator seeded with ``s0``."""
    return int(_load().normgen_splitmix64_output(s0, k))


def bf16_bits(a) -> np.ndarray:
    """bfloat16 encodings (uint16) of finite float32 values, rounded to nearest even:
    the upper 16 bits of the float32 encoding after adding 0x7FFF plus the lowest kept bit."""
    u = np.ascontiguousarray(a, dtype=np.float32).reshape(-1).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_to_f32(h) -> np.ndarray:
    """float32 values of bfloat16 encodings (exact)."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_bf16(a) -> np.ndarray:
    """float32 values rounded to the nearest bfloat16 (ties to even), as float32."""
    return bf16_to_f32(bf16_bits(a))
