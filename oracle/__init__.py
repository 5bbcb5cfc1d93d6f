"""TEST INFRASTRUCTURE: the plain CPU float64 oracle for the three normalizations.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The CUDA library never imports it and
shares no code with it; the only thing the two sides share is the seeded input
generator in ``normgen``.

The arithmetic lives in ``norm_oracle.c`` (plain C, float64, two-pass variance,
one rounding to float32 at the end); its header cites the passage of the pages
each function follows.  This module compiles it with gcc and marshals numpy
arrays through ctypes.

Parity status: every function here is pinned (exact rational brute force,
closed forms, invariants, float64 torch.nn.functional as a third voice, and
planted-mistake runs), see ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "norm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_default = None


def _compile(src_path: str, out_path: str) -> None:
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out_path))
    os.close(fd)
    base = ["gcc", "-O2", "-fPIC", "-shared", "-o", tmp, src_path, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)  # no OpenMP: units run one after another
    os.replace(tmp, out_path)


def build(force: bool = False) -> str:
    """Compile norm_oracle.c into ``oracle/_build/liboracle.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        _compile(SOURCE, _LIB)
    return _LIB


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f32(a, name):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _opt_f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data


class Oracle:
    """ctypes view of one compiled oracle library (the real one, or a planted-mistake build)."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        vp, i64, dbl, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_int
        lib.oracle_layer_norm.restype = ci
        lib.oracle_layer_norm.argtypes = [vp, vp, vp, i64, i64, dbl, vp, vp, ci]
        lib.oracle_rms_channel.restype = ci
        lib.oracle_rms_channel.argtypes = [vp, i64, i64, i64, dbl, vp, vp, ci]
        lib.oracle_group_lrelu_x2.restype = ci
        lib.oracle_group_lrelu_x2.argtypes = [vp, vp, vp, i64, i64, i64, dbl, dbl, vp, vp, ci]
        lib.oracle_group_lrelu_x2_nchw.restype = ci
        lib.oracle_group_lrelu_x2_nchw.argtypes = [vp, vp, vp, i64, i64, i64, i64, dbl, dbl, vp, vp, ci]
        lib.oracle_linear_group_lrelu_x2.restype = ci
        lib.oracle_linear_group_lrelu_x2.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, dbl, dbl, vp, vp, ci]
        self._lib = lib

    @staticmethod
    def _outputs(shape, want64):
        y64 = np.empty(shape, dtype=np.float64) if want64 else None
        y32 = None if want64 else np.empty(shape, dtype=np.float32)
        return y64, y32

    def layer_norm(self, x, gamma, beta, rows, row_len, eps=1e-5, *, f64=False, threads=None):
        """y[r][i] = (x - mean_r) / sqrt(var_r + eps) * gamma[i] + beta[i] over rows of ``row_len``."""
        x = _f32(x, "x")
        if x.size != rows * row_len:
            raise ValueError("x has the wrong size")
        g, b = _opt_f32(gamma), _opt_f32(beta)
        y64, y32 = self._outputs(x.shape, f64)
        rc = self._lib.oracle_layer_norm(_ptr(x), _ptr(g), _ptr(b), rows, row_len, eps,
                                         _ptr(y64), _ptr(y32), threads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_layer_norm rejected its arguments ({rc})")
        return y64 if f64 else y32

    def rms_channel(self, x, B, C, S, eps=1e-5, *, f64=False, threads=None):
        """y[b][c][s] = x[b][c][s] / sqrt(mean_c x[b][:][s]^2 + eps)."""
        x = _f32(x, "x")
        if x.size != B * C * S:
            raise ValueError("x has the wrong size")
        y64, y32 = self._outputs(x.shape, f64)
        rc = self._lib.oracle_rms_channel(_ptr(x), B, C, S, eps, _ptr(y64), _ptr(y32),
                                          threads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_rms_channel rejected its arguments ({rc})")
        return y64 if f64 else y32

    def group_lrelu_x2(self, x, gamma, beta, N, C, G, eps=1e-5, slope=0.01, *, f64=False,
                       threads=None):
        """2 * LeakyReLU(GroupNorm(x)) with G groups of C/G contiguous channels."""
        x = _f32(x, "x")
        if x.size != N * C:
            raise ValueError("x has the wrong size")
        g, b = _opt_f32(gamma), _opt_f32(beta)
        y64, y32 = self._outputs(x.shape, f64)
        rc = self._lib.oracle_group_lrelu_x2(_ptr(x), _ptr(g), _ptr(b), N, C, G, eps, slope,
                                             _ptr(y64), _ptr(y32), threads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_group_lrelu_x2 rejected its arguments ({rc})")
        return y64 if f64 else y32


    def group_lrelu_x2_nchw(self, x, gamma, beta, N, C, S, G, eps=1e-5, slope=0.01, *, f64=False,
                            threads=None):
        """2 * LeakyReLU(GroupNorm(x)) over x[N][C][S]: G groups of C/G contiguous channels,
        each over all S spatial positions."""
        x = _f32(x, "x")
        if x.size != N * C * S:
            raise ValueError("x has the wrong size")
        g, b = _opt_f32(gamma), _opt_f32(beta)
        y64, y32 = self._outputs(x.shape, f64)
        rc = self._lib.oracle_group_lrelu_x2_nchw(_ptr(x), _ptr(g), _ptr(b), N, C, S, G, eps, slope,
                                                  _ptr(y64), _ptr(y32), threads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_group_lrelu_x2_nchw rejected its arguments ({rc})")
        return y64 if f64 else y32


    def linear_group_lrelu_x2(self, x, w, bias, gamma, beta, Mr, K, N, G, eps=1e-5, slope=0.01, *, f64=False,
                              threads=None):
        """2 * LeakyReLU(GroupNorm(x W^T + bias)): x [Mr][K], W [N][K] (nn.Linear's layout), bias
        gamma, beta [N] (or None); G groups of N/G contiguous channels."""
        x = _f32(x, "x")
        w = _f32(w, "w")
        if x.size != Mr * K or w.size != N * K:
            raise ValueError("x or w has the wrong size")
        bb, g, b = _opt_f32(bias), _opt_f32(gamma), _opt_f32(beta)
        y64, y32 = self._outputs((Mr * N,), f64)
        rc = self._lib.oracle_linear_group_lrelu_x2(_ptr(x), _ptr(w), _ptr(bb), _ptr(g), _ptr(b), Mr, K, N, G, eps,
                                                    slope, _ptr(y64), _ptr(y32), threads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_linear_group_lrelu_x2 rejected its arguments ({rc})")
        return y64 if f64 else y32


def get() -> Oracle:
    """The oracle built from ``norm_oracle.c`` as committed."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def build_variant(source_text: str, workdir: str) -> Oracle:
    """Compile a modified copy of the oracle source (used to plant mistakes in tests)."""
    tag = hashlib.sha1(source_text.encode()).hexdigest()[:12]
    src = os.path.join(workdir, f"oracle_{tag}.c")
    with open(src, "w") as f:
        f.write(source_text)
    out = os.path.join(workdir, f"liboracle_{tag}.so")
    _compile(src, out)
    return Oracle(out)


def layer_norm(*a, **k):
    return get().layer_norm(*a, **k)


def rms_channel(*a, **k):
    return get().rms_channel(*a, **k)


def group_lrelu_x2(*a, **k):
    return get().group_lrelu_x2(*a, **k)


def group_lrelu_x2_nchw(*a, **k):
    return get().group_lrelu_x2_nchw(*a, **k)


def linear_group_lrelu_x2(*a, **k):
    return get().linear_group_lrelu_x2(*a, **k)
