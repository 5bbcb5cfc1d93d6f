"""The C ABI on the CPU: the library builds, loads, exports every function that
include/norm.h declares, and rejects bad arguments before touching CUDA.

No call here reaches a kernel: each one fails validation, which happens before
any CUDA runtime call, or is a no-op on empty extents.
"""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "norm.h")

OK, INVALID, MISALIGNED, WORKSPACE = 0, 1, 2, 3


def _build_module():
    import __graft_entry__
    return __graft_entry__._build_module()


@pytest.fixture(scope="module")
def lib():
    _build_module().build()
    import memory_bound_normalization_norm_gb300 as ng
    return ng


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(norm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_operations():
    names = declared_functions()
    for fn in ("norm_layer_fwd", "norm_rms_channel_fwd", "norm_group_lrelu_x2_fwd", "norm_group_lrelu_x2_nchw_fwd"):
        assert fn in names


def test_every_declared_function_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    names = declared_functions()
    missing = [n for n in names if not hasattr(so, n)]
    assert not missing, f"declared in norm.h but not exported: {missing}"
    assert sorted(lib.EXPORTED) == names


def test_library_is_sm103a_only(lib):
    # The build targets exactly one architecture.
    assert _build_module().ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    raw = lib.raw()
    for code, name in [(0, "NORM_OK"), (1, "NORM_ERR_INVALID_ARG"), (2, "NORM_ERR_MISALIGNED"),
                       (3, "NORM_ERR_WORKSPACE"), (4, "NORM_ERR_CUDA"), (5, "NORM_ERR_TIMEOUT"),
                       (6, "NORM_ERR_UNSUPPORTED")]:
        assert raw.norm_status_string(code).decode() == name


def test_options_validate_and_round_trip(lib):
    raw = lib.raw()
    assert raw.norm_set_option(99, 1) == INVALID
    assert raw.norm_set_option(lib.NORM_OPT_LN_PATH, 5) == INVALID
    for path in (4, 3, 2, 1, 0):
        assert raw.norm_set_option(lib.NORM_OPT_LN_PATH, path) == OK
        assert raw.norm_get_option(lib.NORM_OPT_LN_PATH) == path
    assert raw.norm_set_option(lib.NORM_OPT_LN_PATH, -1) == INVALID
    assert raw.norm_set_option(lib.NORM_OPT_BARRIER_TIMEOUT_NS, 0) == INVALID
    old = raw.norm_get_option(lib.NORM_OPT_BARRIER_TIMEOUT_NS)
    assert old == 200_000_000
    assert raw.norm_set_option(lib.NORM_OPT_BARRIER_TIMEOUT_NS, 12345) == OK
    assert raw.norm_get_option(lib.NORM_OPT_BARRIER_TIMEOUT_NS) == 12345
    assert raw.norm_set_option(lib.NORM_OPT_BARRIER_TIMEOUT_NS, old) == OK
    assert raw.norm_set_option(lib.NORM_OPT_GN_PATH, 7) == INVALID
    for path in (6, 5, 4, 3, 2, 1, 0):
        assert raw.norm_set_option(lib.NORM_OPT_GN_PATH, path) == OK
        assert raw.norm_get_option(lib.NORM_OPT_GN_PATH) == path
    for bad in (3, 5, 12, 32, -1):
        assert raw.norm_set_option(lib.NORM_OPT_GN_CLUSTER, bad) == INVALID
    for cl in (16, 8, 4, 2, 1, 0):
        assert raw.norm_set_option(lib.NORM_OPT_GN_CLUSTER, cl) == OK
        assert raw.norm_get_option(lib.NORM_OPT_GN_CLUSTER) == cl


# Fake, well-aligned device addresses: validation must reject before any use.
X, Y, G, B, W = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000


def test_layer_norm_argument_errors(lib):
    f = lib.raw().norm_layer_fwd
    assert f(X, G, B, Y, -1, 16, 1e-5, None, 0, None) == INVALID
    assert f(X, G, B, Y, 2, -16, 1e-5, None, 0, None) == INVALID
    assert f(X, G, B, Y, 2, 16, float("nan"), None, 0, None) == INVALID
    assert f(X, G, B, Y, 2, 16, -1.0, None, 0, None) == INVALID
    assert f(X, G, B, Y, 2, 16, math.inf, None, 0, None) == INVALID
    assert f(None, G, B, Y, 2, 16, 1e-5, None, 0, None) == INVALID
    assert f(X, G, B, None, 2, 16, 1e-5, None, 0, None) == INVALID
    assert f(X + 2, G, B, Y, 2, 16, 1e-5, None, 0, None) == MISALIGNED
    assert f(X, G + 1, B, Y, 2, 16, 1e-5, None, 0, None) == MISALIGNED
    # y partially overlapping x (exact aliasing is allowed), y overlapping gamma
    assert f(X, G, B, X + 4, 2, 16, 1e-5, None, 0, None) == INVALID
    assert f(X, G, B, G + 8, 2, 16, 1e-5, None, 0, None) == INVALID
    # misaligned workspace, workspace overlapping y
    assert f(X, G, B, Y, 2, 16, 1e-5, W + 16, 4096, None) == WORKSPACE
    assert f(X, G, B, Y, 2, 16, 1e-5, Y, 4096, None) == WORKSPACE
    # extents overflowing 2^60 bytes
    assert f(X, G, B, Y, 1 << 40, 1 << 40, 1e-5, None, 0, None) == INVALID
    # empty extents are no-ops, even with null pointers
    assert f(None, None, None, None, 0, 16, 1e-5, None, 0, None) == OK
    assert f(None, None, None, None, 5, 0, 1e-5, None, 0, None) == OK


def test_rms_argument_errors(lib):
    f = lib.raw().norm_rms_channel_fwd
    assert f(X, Y, -1, 4, 4, 1e-5, None) == INVALID
    assert f(X, Y, 1, 4, 4, float("nan"), None) == INVALID
    assert f(None, Y, 1, 4, 4, 1e-5, None) == INVALID
    assert f(X + 1, Y, 1, 4, 4, 1e-5, None) == MISALIGNED
    assert f(X, X + 4, 1, 4, 4, 1e-5, None) == INVALID
    assert f(None, None, 0, 4, 4, 1e-5, None) == OK
    assert f(None, None, 3, 4, 0, 1e-5, None) == OK


def test_group_norm_argument_errors(lib):
    f = lib.raw().norm_group_lrelu_x2_fwd
    assert f(X, G, B, Y, 4, 16, 3, 1e-5, 0.01, None) == INVALID  # 16 % 3 != 0
    assert f(X, G, B, Y, 4, 16, 0, 1e-5, 0.01, None) == INVALID
    assert f(X, G, B, Y, 4, 16, 4, 1e-5, float("inf"), None) == INVALID
    assert f(X, G, B, Y, 4, 16, 4, -1e-5, 0.01, None) == INVALID
    assert f(None, G, B, Y, 4, 16, 4, 1e-5, 0.01, None) == INVALID
    assert f(X, G, B + 2, Y, 4, 16, 4, 1e-5, 0.01, None) == MISALIGNED
    assert f(X, G, B, B, 4, 16, 4, 1e-5, 0.01, None) == INVALID
    assert f(None, None, None, None, 0, 16, 4, 1e-5, 0.01, None) == OK


def test_group_norm_nchw_argument_errors(lib):
    f = lib.raw().norm_group_lrelu_x2_nchw_fwd
    assert f(X, G, B, Y, 4, 16, 9, 3, 1e-5, 0.01, None, 0, None) == INVALID  # 16 % 3 != 0
    assert f(X, G, B, Y, 4, 16, -9, 4, 1e-5, 0.01, None, 0, None) == INVALID
    assert f(X, G, B, Y, 4, 16, 9, 4, float("nan"), 0.01, None, 0, None) == INVALID
    assert f(X, G, B, Y, 4, 16, 9, 4, 1e-5, float("nan"), None, 0, None) == INVALID
    assert f(X + 2, G, B, Y, 4, 16, 9, 4, 1e-5, 0.01, None, 0, None) == MISALIGNED
    # y overlapping x (not exactly), y overlapping beta
    assert f(X, G, B, X + 64, 4, 16, 9, 4, 1e-5, 0.01, None, 0, None) == INVALID
    assert f(X, G, B, B - 8, 4, 16, 9, 4, 1e-5, 0.01, None, 0, None) == INVALID
    # a workspace overlapping y, or not 16-byte aligned
    assert f(X, G, B, Y, 4, 16, 9, 4, 1e-5, 0.01, Y + 64, 4096, None) == WORKSPACE
    assert f(X, G, B, Y, 4, 16, 9, 4, 1e-5, 0.01, W + 8, 4096, None) == WORKSPACE
    # N * C * S overflowing 2^60
    assert f(X, G, B, Y, 1 << 30, 1 << 20, 1 << 20, 4, 1e-5, 0.01, None, 0, None) == INVALID
    assert f(None, None, None, None, 4, 16, 0, 4, 1e-5, 0.01, None, 0, None) == OK
    assert lib.raw().norm_group_lrelu_x2_nchw_fwd_bf16(X + 1, G, B, Y, 4, 16, 9, 4, 1e-5, 0.01, None, 0,
                                                        None) == MISALIGNED
    assert lib.norm_group_lrelu_x2_nchw_workspace_bytes(0, 16, 9, 4) == 0
    assert lib.norm_group_lrelu_x2_nchw_workspace_bytes(4, 16, 9, 3) == 0


def test_workspace_reset_rejects_bad_arguments(lib):
    raw = lib.raw()
    assert raw.norm_layer_workspace_reset(None, 4096, None) == INVALID
    assert raw.norm_layer_workspace_reset(W, 16, None) == INVALID


def test_package_refuses_to_import_without_library(tmp_path):
    # The product path has no CPU fallback: a package copy without the .so must not import.
    import shutil
    import subprocess
    import sys
    pkg = os.path.join(ROOT, "memory_bound_normalization_norm_gb300")
    dst = tmp_path / "memory_bound_normalization_norm_gb300"
    shutil.copytree(pkg, dst, ignore=shutil.ignore_patterns("*.so", "_build", "__pycache__"))
    r = subprocess.run([sys.executable, "-c", "import memory_bound_normalization_norm_gb300"],
                       cwd=tmp_path, capture_output=True, text=True)
    assert r.returncode != 0 and "no CPU fallback" in r.stderr
