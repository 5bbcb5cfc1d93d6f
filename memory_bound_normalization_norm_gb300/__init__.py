"""Python binding of libnormgb300.so: reduce-then-apply normalization on GB300 (fp32,
and bf16 storage with fp32 arithmetic).

This module only marshals arguments into the C ABI of ``include/norm.h``; every
step of every operation runs in the library's own CUDA kernels.  There is no CPU
fallback: importing this package fails loudly if the compiled library is missing
(build it with ``memory_bound_normalization_norm_gb300._build.build()``).

Entry points (same names and argument order as the C functions):

* ``norm_layer_fwd(x, gamma, beta, y, rows, row_len, eps, workspace=None, workspace_bytes=0, stream=None)``
* ``norm_layer_fwd_noalloc(x, gamma, beta, y, rows, row_len, eps, stream=None)``
* ``norm_rms_channel_fwd(x, y, B, C, S, eps, stream=None)``
* ``norm_group_lrelu_x2_fwd(x, gamma, beta, y, N, C, num_groups, eps, negative_slope, stream=None)``
* ``norm_group_lrelu_x2_nchw_fwd(x, gamma, beta, y, N, C, S, num_groups, eps, negative_slope,
  workspace=None, workspace_bytes=0, stream=None)``
* ``norm_layer_fwd_bf16``, ``norm_rms_channel_fwd_bf16``, ``norm_group_lrelu_x2_fwd_bf16``,
  ``norm_group_lrelu_x2_nchw_fwd_bf16``: the same arguments with bfloat16 tensors
* ``norm_linear_group_lrelu_x2_fwd(x, w, bias, gamma, beta, y, M, K, N, num_groups, eps,
  negative_slope, stream=None)``: a Linear with GroupNorm + LeakyReLU + x2 in its epilogue
  (bfloat16 x and w, float32 bias/gamma/beta and y)
* ``norm_last_error(stream=None)``, ``norm_layer_workspace_bytes(rows, row_len)``,
  ``norm_group_lrelu_x2_nchw_workspace_bytes(N, C, S, num_groups)``,
  ``norm_layer_workspace_reset(ws, nbytes, stream=None)``, ``norm_set_option``,
  ``norm_get_option``, ``norm_layer_max_resident_row_len()``

Tensor arguments may be ``torch.Tensor`` (CUDA, contiguous, float32 for the fp32
entry points and bfloat16 for the ``_bf16`` ones: their device pointer is passed) or
plain integers holding device addresses; ``None`` is NULL.
``stream=None`` means torch's current CUDA stream.  Non-zero status codes raise
:class:`NormError`.  PyTorch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnormgb300.so")

NORM_OK = 0
NORM_ERR_INVALID_ARG = 1
NORM_ERR_MISALIGNED = 2
NORM_ERR_WORKSPACE = 3
NORM_ERR_CUDA = 4
NORM_ERR_TIMEOUT = 5
NORM_ERR_UNSUPPORTED = 6

NORM_OPT_LN_PATH = 1
NORM_OPT_BARRIER_TIMEOUT_NS = 2
NORM_OPT_BARRIER_EXTRA_ARRIVALS = 3
NORM_OPT_LN_CTAS = 4
NORM_OPT_GN_PATH = 5
NORM_OPT_GN_CLUSTER = 6

# The C functions this binding exposes (every declaration of include/norm.h).
EXPORTED = (
    "norm_layer_workspace_bytes",
    "norm_layer_fwd",
    "norm_layer_fwd_noalloc",
    "norm_layer_workspace_reset",
    "norm_layer_max_resident_row_len",
    "norm_rms_channel_fwd",
    "norm_group_lrelu_x2_fwd",
    "norm_layer_fwd_bf16",
    "norm_rms_channel_fwd_bf16",
    "norm_group_lrelu_x2_fwd_bf16",
    "norm_group_lrelu_x2_nchw_workspace_bytes",
    "norm_group_lrelu_x2_nchw_fwd",
    "norm_group_lrelu_x2_nchw_fwd_bf16",
    "norm_linear_group_lrelu_x2_fwd",
    "norm_last_error",
    "norm_status_string",
    "norm_set_option",
    "norm_get_option",
)


class NormError(RuntimeError):
    """A non-zero norm_status_t returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {_status_string(status)} ({status})")


if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()'). There is no CPU fallback.")

_lib = ctypes.CDLL(LIB_PATH)
_vp, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_int = ctypes.c_int

_lib.norm_layer_workspace_bytes.restype = _sz
_lib.norm_layer_workspace_bytes.argtypes = [_i64, _i64]
_lib.norm_layer_fwd.restype = _int
_lib.norm_layer_fwd.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _f32, _vp, _sz, _vp]
_lib.norm_layer_fwd_noalloc.restype = _int
_lib.norm_layer_fwd_noalloc.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _f32, _vp]
_lib.norm_layer_workspace_reset.restype = _int
_lib.norm_layer_workspace_reset.argtypes = [_vp, _sz, _vp]
_lib.norm_layer_max_resident_row_len.restype = _i64
_lib.norm_layer_max_resident_row_len.argtypes = []
_lib.norm_rms_channel_fwd.restype = _int
_lib.norm_rms_channel_fwd.argtypes = [_vp, _vp, _i64, _i64, _i64, _f32, _vp]
_lib.norm_group_lrelu_x2_fwd.restype = _int
_lib.norm_group_lrelu_x2_fwd.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _f32, _f32, _vp]
_lib.norm_layer_fwd_bf16.restype = _int
_lib.norm_layer_fwd_bf16.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _f32, _vp, _sz, _vp]
_lib.norm_rms_channel_fwd_bf16.restype = _int
_lib.norm_rms_channel_fwd_bf16.argtypes = [_vp, _vp, _i64, _i64, _i64, _f32, _vp]
_lib.norm_group_lrelu_x2_fwd_bf16.restype = _int
_lib.norm_group_lrelu_x2_fwd_bf16.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _f32, _f32, _vp]
_lib.norm_group_lrelu_x2_nchw_workspace_bytes.restype = _sz
_lib.norm_group_lrelu_x2_nchw_workspace_bytes.argtypes = [_i64, _i64, _i64, _i64]
for _name in ("norm_group_lrelu_x2_nchw_fwd", "norm_group_lrelu_x2_nchw_fwd_bf16"):
    getattr(_lib, _name).restype = _int
    getattr(_lib, _name).argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _f32, _f32, _vp, _sz, _vp]
_lib.norm_linear_group_lrelu_x2_fwd.restype = _int
_lib.norm_linear_group_lrelu_x2_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _f32, _f32, _vp]
_lib.norm_last_error.restype = _int
_lib.norm_last_error.argtypes = [_vp]
_lib.norm_status_string.restype = ctypes.c_char_p
_lib.norm_status_string.argtypes = [_int]
_lib.norm_set_option.restype = _int
_lib.norm_set_option.argtypes = [_int, _i64]
_lib.norm_get_option.restype = _i64
_lib.norm_get_option.argtypes = [_int]


def _status_string(status: int) -> str:
    return _lib.norm_status_string(int(status)).decode()


def _ptr(a, bf16: bool = False):
    """Device address of a tensor argument (None -> NULL)."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    dt = getattr(a, "dtype", None)
    if dt is not None and hasattr(a, "data_ptr"):
        import torch
        want = torch.bfloat16 if bf16 else torch.float32
        if a.dtype != want and a.dtype != torch.uint8:
            raise TypeError(f"expected a {want} tensor, got {a.dtype}")
        if not a.is_cuda:
            raise TypeError("expected a CUDA tensor (the library takes device pointers)")
        if not a.is_contiguous():
            raise TypeError("expected a contiguous tensor")
        return a.data_ptr()
    raise TypeError(f"cannot pass {type(a).__name__} as a device pointer")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str) -> None:
    if status != NORM_OK:
        raise NormError(status, where)


# ------------------------------------------------------------------ C entry points

def norm_layer_workspace_bytes(rows: int, row_len: int) -> int:
    return int(_lib.norm_layer_workspace_bytes(rows, row_len))


def norm_layer_max_resident_row_len() -> int:
    return int(_lib.norm_layer_max_resident_row_len())


def norm_layer_fwd(x, gamma, beta, y, rows, row_len, eps, workspace=None, workspace_bytes=0, stream=None):
    _check(_lib.norm_layer_fwd(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), rows, row_len, eps,
                               _ptr(workspace), workspace_bytes, _stream(stream)), "norm_layer_fwd")


def norm_layer_fwd_noalloc(x, gamma, beta, y, rows, row_len, eps, stream=None):
    """LayerNorm whose scratch is a fixed 1 MiB array inside the library, for callers
    that cannot allocate device memory; see include/norm.h for its limits."""
    _check(_lib.norm_layer_fwd_noalloc(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), rows, row_len, eps,
                                       _stream(stream)), "norm_layer_fwd_noalloc")


def norm_layer_workspace_reset(workspace, workspace_bytes, stream=None):
    _check(_lib.norm_layer_workspace_reset(_ptr(workspace), workspace_bytes, _stream(stream)),
           "norm_layer_workspace_reset")


def norm_rms_channel_fwd(x, y, B, C, S, eps, stream=None):
    _check(_lib.norm_rms_channel_fwd(_ptr(x), _ptr(y), B, C, S, eps, _stream(stream)), "norm_rms_channel_fwd")


def norm_group_lrelu_x2_fwd(x, gamma, beta, y, N, C, num_groups, eps, negative_slope, stream=None):
    _check(_lib.norm_group_lrelu_x2_fwd(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), N, C, num_groups, eps,
                                        negative_slope, _stream(stream)), "norm_group_lrelu_x2_fwd")


def norm_layer_fwd_bf16(x, gamma, beta, y, rows, row_len, eps, workspace=None, workspace_bytes=0, stream=None):
    _check(_lib.norm_layer_fwd_bf16(_ptr(x, True), _ptr(gamma, True), _ptr(beta, True), _ptr(y, True), rows,
                                    row_len, eps, _ptr(workspace), workspace_bytes, _stream(stream)),
           "norm_layer_fwd_bf16")


def norm_rms_channel_fwd_bf16(x, y, B, C, S, eps, stream=None):
    _check(_lib.norm_rms_channel_fwd_bf16(_ptr(x, True), _ptr(y, True), B, C, S, eps, _stream(stream)),
           "norm_rms_channel_fwd_bf16")


def norm_group_lrelu_x2_fwd_bf16(x, gamma, beta, y, N, C, num_groups, eps, negative_slope, stream=None):
    _check(_lib.norm_group_lrelu_x2_fwd_bf16(_ptr(x, True), _ptr(gamma, True), _ptr(beta, True), _ptr(y, True), N,
                                             C, num_groups, eps, negative_slope, _stream(stream)),
           "norm_group_lrelu_x2_fwd_bf16")


def norm_group_lrelu_x2_nchw_workspace_bytes(N: int, C: int, S: int, num_groups: int) -> int:
    return int(_lib.norm_group_lrelu_x2_nchw_workspace_bytes(N, C, S, num_groups))


def norm_group_lrelu_x2_nchw_fwd(x, gamma, beta, y, N, C, S, num_groups, eps, negative_slope, workspace=None,
                                 workspace_bytes=0, stream=None):
    _check(_lib.norm_group_lrelu_x2_nchw_fwd(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), N, C, S, num_groups, eps,
                                             negative_slope, _ptr(workspace), workspace_bytes, _stream(stream)),
           "norm_group_lrelu_x2_nchw_fwd")


def norm_group_lrelu_x2_nchw_fwd_bf16(x, gamma, beta, y, N, C, S, num_groups, eps, negative_slope, workspace=None,
                                      workspace_bytes=0, stream=None):
    _check(_lib.norm_group_lrelu_x2_nchw_fwd_bf16(_ptr(x, True), _ptr(gamma, True), _ptr(beta, True),
                                                  _ptr(y, True), N, C, S, num_groups, eps, negative_slope,
                                                  _ptr(workspace), workspace_bytes, _stream(stream)),
           "norm_group_lrelu_x2_nchw_fwd_bf16")


def norm_linear_group_lrelu_x2_fwd(x, w, bias, gamma, beta, y, M, K, N, num_groups, eps, negative_slope,
                                   stream=None):
    """2 * LeakyReLU(GroupNorm(x W^T + bias)) in one kernel: x [M][K] and w [N][K] bfloat16,
    bias/gamma/beta [N] and y [M][N] float32."""
    _check(_lib.norm_linear_group_lrelu_x2_fwd(_ptr(x, True), _ptr(w, True), _ptr(bias), _ptr(gamma), _ptr(beta),
                                               _ptr(y), M, K, N, num_groups, eps, negative_slope, _stream(stream)),
           "norm_linear_group_lrelu_x2_fwd")


def norm_last_error(stream=None) -> int:
    """Synchronize the stream; return (and clear) the device error word as a status code."""
    return int(_lib.norm_last_error(_stream(stream)))


def norm_status_string(status: int) -> str:
    return _status_string(status)


def norm_set_option(option: int, value: int) -> None:
    _check(_lib.norm_set_option(option, value), "norm_set_option")


def norm_get_option(option: int) -> int:
    return int(_lib.norm_get_option(option))


# ------------------------------------------------------------------ raw status forms

def raw():
    """The ctypes library handle, for callers that want status codes instead of exceptions."""
    return _lib


# ------------------------------------------------------------------ tensor conveniences

def layer_norm(x, gamma=None, beta=None, eps: float = 1e-5, normalized_ndim: int | None = None, out=None,
               stream=None):
    """LayerNorm of a CUDA float32 or bfloat16 tensor over its last ``normalized_ndim``
    dims (default: the dims of ``gamma``, else all but the first); gamma/beta of the
    same dtype."""
    import torch
    if normalized_ndim is None:
        normalized_ndim = gamma.dim() if gamma is not None else x.dim() - 1
    row_len = 1
    for d in x.shape[x.dim() - normalized_ndim:]:
        row_len *= int(d)
    rows = x.numel() // row_len if row_len else 0
    y = torch.empty_like(x) if out is None else out
    fn = norm_layer_fwd_bf16 if x.dtype == torch.bfloat16 else norm_layer_fwd
    fn(x, gamma, beta, y, rows, row_len, eps, stream=stream)
    return y


def rms_norm_channel(x, eps: float = 1e-5, out=None, stream=None):
    """RMSNorm over dim 1 of a CUDA float32 or bfloat16 tensor of shape (B, C, *spatial)."""
    import torch
    B, C = int(x.shape[0]), int(x.shape[1])
    S = x.numel() // (B * C) if B * C else 0
    y = torch.empty_like(x) if out is None else out
    fn = norm_rms_channel_fwd_bf16 if x.dtype == torch.bfloat16 else norm_rms_channel_fwd
    fn(x, y, B, C, S, eps, stream=stream)
    return y


def group_norm_lrelu_x2(x, num_groups: int, gamma=None, beta=None, eps: float = 1e-5,
                        negative_slope: float = 0.01, out=None, stream=None):
    """2 * LeakyReLU(GroupNorm(x)) for a CUDA float32 or bfloat16 tensor of shape (N, C) or
    (N, C, *spatial); a group spans its channels at every spatial position."""
    import torch
    N, C = int(x.shape[0]), int(x.shape[1])
    y = torch.empty_like(x) if out is None else out
    bf16 = x.dtype == torch.bfloat16
    if x.dim() == 2:
        fn = norm_group_lrelu_x2_fwd_bf16 if bf16 else norm_group_lrelu_x2_fwd
        fn(x, gamma, beta, y, N, C, num_groups, eps, negative_slope, stream=stream)
    else:
        S = x.numel() // (N * C) if N * C else 0
        fn = norm_group_lrelu_x2_nchw_fwd_bf16 if bf16 else norm_group_lrelu_x2_nchw_fwd
        fn(x, gamma, beta, y, N, C, S, num_groups, eps, negative_slope, stream=stream)
    return y
