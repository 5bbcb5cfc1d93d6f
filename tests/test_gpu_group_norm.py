"""GroupNorm + LeakyReLU + x2 on the GPU against the float64 oracle, element by element.

Covers the vector kernel (M = 4..128, powers of two) at ragged and wide shapes, the
team-per-group kernel (M = 1, 2, 3, 48, 256 and other sizes up to 1,024, misaligned
pointers), NULL affine, in-place, slopes, and the full-size (1024, 8192), 512-group
workload.
"""
import numpy as np
import pytest

import normgen
import oracle
from gpu_util import Guarded, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ng():
    import memory_bound_normalization_norm_gb300 as m
    return m


def run_gn(ng, x, g, b, N, C, G, eps=1e-5, slope=0.01, offset=0, inplace=False):
    xb = Guarded(N * C, x, offset=offset)
    gd = None if g is None else Guarded(C, g, offset=offset).t
    bd = None if b is None else Guarded(C, b, offset=offset).t
    yb = xb if inplace else Guarded(N * C, offset=offset)
    ng.norm_group_lrelu_x2_fwd(xb.t, gd, bd, yb.t, N, C, G, eps, slope)
    out = yb.numpy()
    assert yb.guards_intact(), "GroupNorm wrote outside its output"
    return out


def inputs(N, C, seed, affine=True):
    x = normgen.normal(N * C, seed=seed, tensor_id=0)
    if not affine:
        return x, None, None
    return x, normgen.normal(C, 1.0, 0.1, seed=seed, tensor_id=1), normgen.normal(C, 0.0, 0.1, seed=seed, tensor_id=2)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 16, 32, 48, 64, 128, 256])
@pytest.mark.parametrize("N,G", [(1, 1), (7, 5), (33, 16)])
def test_group_sizes(ng, M, N, G):
    C = M * G
    x, g, b = inputs(N, C, seed=M * 100 + G)
    want = oracle.group_lrelu_x2(x, g, b, N, C, G)
    assert_parity(run_gn(ng, x, g, b, N, C, G), want, f"GN N={N} C={C} G={G}")


@pytest.mark.parametrize("slope", [0.0, 0.01, 0.2, 1.0, -0.5])
def test_slopes(ng, slope):
    N, C, G = 9, 1024, 64
    x, g, b = inputs(N, C, seed=4)
    want = oracle.group_lrelu_x2(x, g, b, N, C, G, slope=slope)
    assert_parity(run_gn(ng, x, g, b, N, C, G, slope=slope), want, f"GN slope={slope}")


@pytest.mark.parametrize("M", [16, 3])
def test_no_affine_in_place_and_misaligned(ng, M):
    N, G = 17, 24
    C = M * G
    x, _, _ = inputs(N, C, seed=8, affine=False)
    want = oracle.group_lrelu_x2(x, None, None, N, C, G)
    assert_parity(run_gn(ng, x, None, None, N, C, G), want, "GN no affine")
    assert_parity(run_gn(ng, x, None, None, N, C, G, inplace=True), want, "GN in place")
    x, g, b = inputs(N, C, seed=9)
    want = oracle.group_lrelu_x2(x, g, b, N, C, G)
    assert_parity(run_gn(ng, x, g, b, N, C, G, offset=1), want, "GN misaligned")


def test_one_channel_per_group_is_two_lrelu_beta(ng):
    # The worked case on the GroupNorm page: M = 1 gives 2 * LeakyReLU(beta) exactly.
    N, C = 5, 64
    x, g, b = inputs(N, C, seed=12)
    got = run_gn(ng, x, g, b, N, C, C).reshape(N, C)
    bd = b.astype(np.float32)
    want = 2.0 * np.where(bd > 0, bd, np.float32(0.01) * bd)
    assert np.array_equal(got, np.tile(want.astype(np.float32), (N, 1)))


def test_full_size(ng):
    """(1024, 8192), 512 groups of 16 channels, gamma ~ N(1, 0.1), beta ~ N(0, 0.1), slope 0.01."""
    N, C, G = 1024, 8192, 512
    x, g, b = inputs(N, C, seed=0)
    want = oracle.group_lrelu_x2(x, g, b, N, C, G)
    assert_parity(run_gn(ng, x, g, b, N, C, G), want, "GN full size")


def test_many_rows_fold_grid(ng):
    # more rows than one grid dimension holds (65535): rows are folded
    N, C, G = 70000, 16, 1
    x, g, b = inputs(N, C, seed=13)
    assert_parity(run_gn(ng, x, g, b, N, C, G), oracle.group_lrelu_x2(x, g, b, N, C, G), "GN 70000 rows")


@pytest.mark.parametrize("N,C,G", [
    (1000, 4104, 513),  # M = 8: a ragged last column block in every row
    (5000, 64, 4),      # rows of 16 float4: most of each column block is out of range
    (3, 12, 3),         # three float4 per row
])
def test_ragged_shapes(ng, N, C, G):
    x, g, b = inputs(N, C, seed=N + C)
    want = oracle.group_lrelu_x2(x, g, b, N, C, G)
    assert_parity(run_gn(ng, x, g, b, N, C, G), want, f"GN N={N} C={C} G={G}")
    assert_parity(run_gn(ng, x, g, b, N, C, G, inplace=True), want, f"GN in place N={N} C={C} G={G}")


def test_wide_rows(ng):
    # 16384 channels: eight column blocks per row
    N, C, G = 9, 16384, 512
    x, g, b = inputs(N, C, seed=21)
    assert_parity(run_gn(ng, x, g, b, N, C, G), oracle.group_lrelu_x2(x, g, b, N, C, G), "GN C=16384")


@pytest.mark.parametrize("N,C,G", [
    (2000, 1536, 32),   # M = 48
    (1000, 1200, 40),   # M = 30: the scalar form
    (500, 3072, 32),    # M = 96
    (300, 6144, 32),    # M = 192
    (100, 1000, 1),     # M = 1000: 250 vectors a group
    (50, 2048, 2),      # M = 1024: the longest team group
    (40, 2052, 2),      # M = 1026: past the team kernel, to the register kernel
])
def test_group_sizes_not_powers_of_two(ng, N, C, G):
    x, g, b = inputs(N, C, seed=N + C + G)
    want = oracle.group_lrelu_x2(x, g, b, N, C, G)
    assert_parity(run_gn(ng, x, g, b, N, C, G), want, f"GN N={N} C={C} G={G}")
    assert_parity(run_gn(ng, x, g, b, N, C, G, offset=1), want, f"GN misaligned N={N} C={C} G={G}")
