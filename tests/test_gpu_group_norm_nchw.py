"""GroupNorm + LeakyReLU + x2 over NCHW tensors on the GPU against the float64 oracle,
element by element.

A group is its M = C/G channels at all S = H*W positions, M*S contiguous values.
Covered: the register kernel with one CTA per group (channel-per-vector, per-element
and S = 1 channel maps), thread-block clusters of 2..16 CTAs (automatic and forced,
ragged slices), its streamed form (bulk copies into double-buffered shared memory,
clusters walking many groups, bounded waits that give up cleanly), the persistent
single-read kernel in its GroupNorm form (row groups, channel maps with S below and above
a CTA's vector stride, a caller workspace shared with the two-kernel path, bounded
waits), the two-kernel path (vector and scalar, caller and library workspace, more
than 65,535 groups), the warp path, NULL affine, in place, misaligned pointers,
cancellation-heavy inputs, and the (8, 512, 64, 64) 32-group workload.
"""
import numpy as np
import pytest

import normgen
import oracle
from gpu_util import Guarded, assert_parity

pytestmark = pytest.mark.gpu

REG, SPLIT, WARP, STREAM, TEAM, PERS = 1, 2, 3, 4, 5, 6


@pytest.fixture(scope="module")
def ng():
    import memory_bound_normalization_norm_gb300 as m
    yield m
    m.norm_set_option(m.NORM_OPT_GN_PATH, 0)
    m.norm_set_option(m.NORM_OPT_GN_CLUSTER, 0)


def inputs(N, C, S, seed, mean=0.0, std=1.0, affine=True):
    x = normgen.normal(N * C * S, mean, std, seed=seed, tensor_id=0)
    if not affine:
        return x, None, None
    return x, normgen.normal(C, 1.0, 0.1, seed=seed, tensor_id=1), normgen.normal(C, 0.0, 0.1, seed=seed, tensor_id=2)


def run(ng, x, g, b, N, C, S, G, path=0, cluster=0, slope=0.01, offset=0, inplace=False, workspace=None,
        ws_bytes=0):
    ng.norm_set_option(ng.NORM_OPT_GN_PATH, path)
    ng.norm_set_option(ng.NORM_OPT_GN_CLUSTER, cluster)
    try:
        n = N * C * S
        xb = Guarded(n, x, offset=offset)
        gd = None if g is None else Guarded(C, g, offset=offset).t
        bd = None if b is None else Guarded(C, b, offset=offset).t
        yb = xb if inplace else Guarded(n, offset=offset)
        ng.norm_group_lrelu_x2_nchw_fwd(xb.t, gd, bd, yb.t, N, C, S, G, 1e-5, slope, workspace, ws_bytes)
        assert ng.norm_last_error() == 0
    finally:
        ng.norm_set_option(ng.NORM_OPT_GN_PATH, 0)
        ng.norm_set_option(ng.NORM_OPT_GN_CLUSTER, 0)
    out = yb.numpy()
    assert yb.guards_intact(), "GroupNorm NCHW wrote outside its output"
    return out


def check(ng, N, C, S, G, seed=0, **kw):
    x, g, b = inputs(N, C, S, seed)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, slope=kw.get("slope", 0.01), f64=True)
    assert_parity(run(ng, x, g, b, N, C, S, G, **kw), want, f"GN NCHW ({N},{C},{S})/{G} {kw}")


# ------------------------------------------------------------------ register kernel, one CTA per group

@pytest.mark.parametrize("N,C,S,G", [
    (2, 32, 64, 8),     # M = 4, L = 256: one channel per 4-element vector
    (3, 64, 1024, 32),  # L = 2048
    (2, 96, 36, 12),    # L = 288: ragged last vectors of the CTA
    (2, 8, 6, 4),       # S = 6: channels change inside a vector
    (3, 12, 7, 3),      # S = 7, L = 28
    (4, 48, 1, 6),      # S = 1: consecutive channels
    (5, 256, 1, 2),     # S = 1, M = 128
    (1, 16, 512, 2),    # L = 4096: 128 threads x 8 vectors
    (2, 4, 2048, 1),    # L = 8192: a full 256-thread CTA
])
def test_register_kernel(ng, N, C, S, G):
    check(ng, N, C, S, G, seed=N * C + S, path=REG)
    check(ng, N, C, S, G, seed=N * C + S)


# ------------------------------------------------------------------ team kernel (short groups)

@pytest.mark.parametrize("N,C,S,G", [
    (2, 32, 64, 8),      # L = 256: 64 vectors, teams of 16 lanes x 4
    (2, 256, 4, 1),      # L = 1024: 256 vectors, a warp x 8, the longest team group
    (4, 48, 1, 1),       # S = 1, M = 48: 12 vectors, teams of 4 lanes x 3
    (5, 240, 1, 6),      # S = 1, M = 40: 10 vectors, ragged last lane
    (3, 96, 1, 1),       # S = 1, M = 96: 24 vectors, teams of 8 x 3
    (2, 8, 6, 4),        # S = 6: channels change inside a vector (L = 12)
    (3, 12, 7, 3),       # S = 7, L = 28
    (9, 4, 1, 1),        # L = 4: one vector, a team of one lane
    (700, 64, 3, 16),    # 11,200 groups of 12: grid-stride over many teams per CTA
])
def test_team_kernel(ng, N, C, S, G):
    check(ng, N, C, S, G, seed=N * C + S + 7, path=TEAM)
    x, g, b = inputs(N, C, S, seed=N + S)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, f64=True)
    assert_parity(run(ng, x, g, b, N, C, S, G, path=TEAM, inplace=True), want, "GN team in place")


@pytest.mark.parametrize("N,C,S,G", [
    (3, 30, 1, 1),       # M = 30: pairs of elements (L even, not a multiple of 4)
    (5, 18, 3, 3),       # L = 18, S = 3: pairs whose channels differ
    (2, 510, 1, 1),      # L = 510: 255 pairs, a warp x 8
    (2, 9, 5, 3),        # L = 15: one element an item
    (1, 1, 1, 1),        # a group of one value: y = 2 LeakyReLU(beta)
    (2, 256, 1, 1),      # L = 256: vectors here, single elements (256, the most) misaligned
    (4, 32, 2, 4),       # L = 16, misaligned below
])
def test_team_kernel_pair_and_scalar_forms(ng, N, C, S, G):
    # offset 0: 4-element or 2-element items by L; offset 1 (4 bytes): single elements,
    # at most 256 of them
    check(ng, N, C, S, G, seed=N + C + S, path=TEAM)
    if C // G * S <= 256:
        check(ng, N, C, S, G, seed=N + C + S + 1, path=TEAM, offset=1)
    else:
        x, g, b = inputs(N, C, S, seed=1)
        with pytest.raises(ng.NormError) as e:
            run(ng, x, g, b, N, C, S, G, path=TEAM, offset=1)
        assert e.value.status == ng.NORM_ERR_UNSUPPORTED
        check(ng, N, C, S, G, seed=N + C + S + 1, offset=1)  # the automatic choice serves it


def test_team_kernel_no_affine(ng):
    N, C, S, G = 6, 96, 2, 4
    x, _, _ = inputs(N, C, S, seed=61, affine=False)
    want = oracle.group_lrelu_x2_nchw(x, None, None, N, C, S, G, f64=True)
    assert_parity(run(ng, x, None, None, N, C, S, G, path=TEAM), want, "GN team no affine")


def test_team_kernel_refuses_long_groups(ng):
    x, g, b = inputs(1, 4, 260, seed=62)  # L = 1040: 260 vectors
    with pytest.raises(ng.NormError) as e:
        run(ng, x, g, b, 1, 4, 260, 1, path=TEAM)
    assert e.value.status == ng.NORM_ERR_UNSUPPORTED
    x, g, b = inputs(1, 4, 65, seed=62)  # L = 260 elements, misaligned: the scalar form holds 256
    with pytest.raises(ng.NormError) as e:
        run(ng, x, g, b, 1, 4, 65, 1, path=TEAM, offset=1)
    assert e.value.status == ng.NORM_ERR_UNSUPPORTED


# ------------------------------------------------------------------ clusters

@pytest.mark.parametrize("cluster", [0, 2, 4, 8, 16])
@pytest.mark.parametrize("N,C,S,G", [
    (2, 64, 1024, 4),   # L = 16384: automatic cluster of 2
    (1, 3, 2732, 1),    # L = 8196: slices of 1025 and 1024 vectors, S % 4 != 0
    (3, 32, 1000, 8),   # L = 4000
])
def test_clusters(ng, cluster, N, C, S, G):
    check(ng, N, C, S, G, seed=cluster + S, path=REG, cluster=cluster)


def test_cluster_of_sixteen_at_capacity(ng):
    # L = 131072, the longest group the register kernel holds: 16 CTAs of 8192
    check(ng, 2, 32, 16384, 4, seed=5)


def test_cluster_ragged_empty_ranks(ng):
    # L = 20 (5 vectors) over 8 CTAs: three ranks hold nothing and still take part
    check(ng, 3, 20, 4, 4, seed=6, path=REG, cluster=8)


def test_full_size(ng):
    """(8, 512, 64, 64), 32 groups: groups of 16 channels x 4096 positions, L = 65536."""
    check(ng, 8, 512, 4096, 32, seed=0)


# ------------------------------------------------------------------ streamed register kernel

@pytest.mark.parametrize("N,C,S,G,cluster", [
    (3, 64, 1024, 32, 1),    # L = 2048: 512-vector slices, 4 vectors a thread
    (2, 4, 2048, 1, 1),      # L = 8192: 2048-vector slices, 8 vectors a thread
    (64, 64, 1024, 16, 1),   # 1024 groups: every CTA walks many groups through both buffers
    (2, 64, 1024, 4, 2),     # L = 16384 over clusters of 2 .. 16
    (2, 64, 1024, 4, 4),
    (2, 64, 1024, 4, 8),
    (2, 64, 1024, 4, 16),
    (1, 3, 2732, 1, 2),      # L = 8196: slices of 1026 and 1023 vectors
    (5, 8192, 1, 2, 1),      # S = 1: consecutive channels
    (2, 8, 2046, 4, 2),      # S = 2046: channels change inside a vector
    (40, 256, 1024, 8, 4),   # 320 groups over clusters of 4
    (3, 64, 300, 2, 2),      # S = 300 < 4 * NT: a thread's step is 3 channels and 124 values
    (2, 16, 1020, 1, 2),     # S = 1020: a step is 1 channel and 4 values
    (4, 32, 516, 2, 0),      # S = 516, automatic cluster
    (160, 32, 2048, 4, 2),   # S = 2048 >= 4 * NT, full slices (the check-free copy), 2-3 groups a cluster
])
def test_streamed(ng, N, C, S, G, cluster):
    check(ng, N, C, S, G, seed=N + C + S + cluster, path=STREAM, cluster=cluster)


@pytest.mark.parametrize("N,C,S,G", [
    (8, 512, 2048, 32),    # 256 groups of 32,768: split over 8 CTAs of 1,024 vectors, not 4 of 2,048
    (16, 512, 2048, 32),   # 512 groups of 32,768: the same
    (32, 512, 1024, 32),   # 1,024 groups of 16,384: split over 4 CTAs, not 2
    (4, 512, 2048, 32),    # 128 groups: the doubled split declined (one wave over clusters of 4)
])
def test_streamed_split_over_twice_the_ctas(ng, N, C, S, G):
    # the automatic choice may split a group over twice the CTAs of the smallest
    # cluster that holds it, when the waves of groups make that faster
    check(ng, N, C, S, G, seed=N + S + 5)


def test_streamed_is_the_automatic_choice_at_full_size(ng):
    # the (8, 512, 64, 64) workload: clusters of 8 CTAs with 2048-vector slices
    N, C, S, G = 8, 512, 4096, 32
    x, g, b = inputs(N, C, S, seed=51)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, f64=True)
    assert_parity(run(ng, x, g, b, N, C, S, G, path=STREAM), want, "GN NCHW streamed full size")
    assert_parity(run(ng, x, g, b, N, C, S, G, path=STREAM, inplace=True), want, "GN NCHW streamed in place")


def test_streamed_tiny_wait_limit_gives_up_cleanly(ng):
    """With a 1 ns limit the CTAs stop waiting for their bulk copies: the call records
    NORM_ERR_TIMEOUT (or finishes, if every copy had landed at its first check), every
    element of y keeps its previous value or holds its correct result, and the next
    call with the default limit is correct."""
    N, C, S, G = 16, 64, 1024, 8
    x, g, b = inputs(N, C, S, seed=52)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, f64=True)
    old = ng.norm_get_option(ng.NORM_OPT_BARRIER_TIMEOUT_NS)
    xb, gb, bb, yb = Guarded(N * C * S, x), Guarded(C, g), Guarded(C, b), Guarded(N * C * S)
    ng.norm_set_option(ng.NORM_OPT_GN_PATH, STREAM)
    ng.norm_set_option(ng.NORM_OPT_BARRIER_TIMEOUT_NS, 1)
    try:
        ng.norm_group_lrelu_x2_nchw_fwd(xb.t, gb.t, bb.t, yb.t, N, C, S, G, 1e-5, 0.01)
        status = ng.norm_last_error()
    finally:
        ng.norm_set_option(ng.NORM_OPT_BARRIER_TIMEOUT_NS, old)
        ng.norm_set_option(ng.NORM_OPT_GN_PATH, 0)
    assert status in (ng.NORM_OK, ng.NORM_ERR_TIMEOUT)
    got = yb.numpy().astype(np.float64)
    untouched = np.isnan(got)  # the guard sentinel is a NaN no kernel writes
    ok = np.abs(got - want) <= 1e-4 * (1.0 + np.abs(want))
    assert np.all(untouched | ok), "an element of y is neither untouched nor correct"
    assert yb.guards_intact()
    assert_parity(run(ng, x, g, b, N, C, S, G, path=STREAM), want, "GN NCHW streamed after a timeout")


# ------------------------------------------------------------------ two-kernel path

@pytest.mark.parametrize("N,C,S,G,path", [
    (1, 128, 65536, 32, SPLIT),  # L = 262144: longer than a 16-CTA cluster holds
    (2, 8, 36000, 2, SPLIT),     # L = 144000
    (3, 12, 7, 3, SPLIT),    # vector form, short groups
    (3, 9, 5, 3, SPLIT),     # scalar form (L = 15)
    (2, 6, 2001, 3, 0),      # scalar form, L = 4002 ... taken by the warp path
    (1, 5, 1001, 1, 0),      # scalar form, L = 5005 > 4096: two-kernel path
])
def test_split(ng, N, C, S, G, path):
    check(ng, N, C, S, G, seed=C + S, path=path)


@pytest.mark.parametrize("N,C,S,G", [(3, 64, 65536, 8), (3, 40, 131072, 5)])
def test_split_large(ng, N, C, S, G):
    # 50 and 60 MB of x through the two-kernel path, groups of 524,288 and
    # 1,048,576 values
    check(ng, N, C, S, G, seed=S + G, path=SPLIT)
    x, g, b = inputs(N, C, S, S + G)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, f64=True)
    assert_parity(run(ng, x, g, b, N, C, S, G, path=SPLIT, inplace=True), want, "GN NCHW large split in place")


def test_split_caller_workspace(ng):
    import torch
    N, C, S, G = 1, 64, 8192, 4
    need = ng.norm_group_lrelu_x2_nchw_workspace_bytes(N, C, S, G)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    check(ng, N, C, S, G, seed=31, path=SPLIT, workspace=ws, ws_bytes=need)
    x, g, b = inputs(N, C, S, 31)
    with pytest.raises(ng.NormError) as e:
        run(ng, x, g, b, N, C, S, G, path=SPLIT, workspace=ws, ws_bytes=16)
    assert e.value.status == ng.NORM_ERR_WORKSPACE


def test_split_many_groups_fold_grid(ng):
    # more groups than one grid dimension holds (65535)
    check(ng, 70000, 4, 2, 1, seed=32, path=SPLIT)


# ------------------------------------------------------------------ persistent kernel, GroupNorm form

@pytest.mark.parametrize("N,C,S,G,path", [
    (1, 128, 65536, 32, PERS), # L = 262144: 32 segments over row groups
    (2, 8, 36000, 2, PERS),    # L = 144000, 4 segments: a row group each
    (1, 4, 262144, 1, PERS),   # L = 1,048,576: one segment over the whole grid
    (2, 6, 65540, 3, PERS),    # L = 131080: S not a multiple of a CTA's vector stride
    (2, 2048, 4, 16, PERS),    # S = 4: a new channel at every vector
    (3, 96, 12, 8, PERS),      # S = 12: a new channel every three vectors
    (64, 64, 4096, 8, PERS),   # 512 segments of 32,768: many segments per row group
    (5, 10, 8, 5, PERS),       # L = 16: fewer vectors than a row group has CTAs
])
def test_persistent(ng, N, C, S, G, path):
    check(ng, N, C, S, G, seed=N + C + S + G, path=path)


@pytest.mark.parametrize("N,C,S,G", [(3, 64, 65536, 8), (3, 40, 131072, 5)])
def test_persistent_large(ng, N, C, S, G):
    # the two-kernel path's large cases (x of 48 and 60 MiB): the automatic choice
    # is the persistent kernel, one read of x
    check(ng, N, C, S, G, seed=S + G + 1)
    x, g, b = inputs(N, C, S, S + G + 1)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, f64=True)
    assert_parity(run(ng, x, g, b, N, C, S, G, inplace=True), want, "GN NCHW persistent in place")


def test_persistent_long_workload(ng):
    """(1, 128, 512, 512), 32 groups: 32 segments of 1,048,576 values."""
    check(ng, 1, 128, 512 * 512, 32, seed=0)


@pytest.mark.parametrize("slope", [0.0, 0.2, 1.0, -0.5])
def test_persistent_slopes_and_no_affine(ng, slope):
    N, C, S, G = 2, 8, 36000, 2
    check(ng, N, C, S, G, seed=72, slope=slope, path=PERS)
    x, _, _ = inputs(N, C, S, seed=73, affine=False)
    want = oracle.group_lrelu_x2_nchw(x, None, None, N, C, S, G, slope=slope, f64=True)
    assert_parity(run(ng, x, None, None, N, C, S, G, slope=slope, path=PERS), want,
                  f"GN persistent no affine {slope}")


def test_persistent_and_split_share_a_caller_workspace(ng):
    """The persistent path keeps its header and records at the start of the workspace and
    the two-kernel path writes its partials after them: calls of both, in any order, on one
    zero-filled workspace stay correct."""
    import torch
    N, C, S, G = 2, 8, 36000, 2
    need = ng.norm_group_lrelu_x2_nchw_workspace_bytes(N, C, S, G)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    x, g, b = inputs(N, C, S, seed=74)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, f64=True)
    for path in (PERS, SPLIT, PERS, 0, SPLIT, SPLIT, PERS):
        assert_parity(run(ng, x, g, b, N, C, S, G, path=path, workspace=ws, ws_bytes=need), want,
                      f"shared workspace path={path}")
    with pytest.raises(ng.NormError) as e:
        run(ng, x, g, b, N, C, S, G, path=PERS, workspace=ws, ws_bytes=64)
    assert e.value.status == ng.NORM_ERR_WORKSPACE


def test_persistent_refusals(ng):
    x, g, b = inputs(2, 6, 2001, seed=75)  # S % 4 != 0: a vector would straddle two channels
    with pytest.raises(ng.NormError) as e:
        run(ng, x, g, b, 2, 6, 2001, 3, path=PERS)
    assert e.value.status == ng.NORM_ERR_UNSUPPORTED
    x, g, b = inputs(2, 16, 64, seed=75)
    with pytest.raises(ng.NormError) as e:
        run(ng, x, g, b, 2, 16, 64, 4, path=PERS, offset=1)  # not 16-byte aligned
    assert e.value.status == ng.NORM_ERR_UNSUPPORTED


def test_persistent_tiny_wait_limit_gives_up_cleanly(ng):
    """With a 1 ns limit the waits that are not over at their first look give up: the call
    records NORM_ERR_TIMEOUT (or finishes), every element of y keeps its previous value or
    holds its correct result, and the next call with the default limit is correct (the
    library's workspace is reset when the timeout is read)."""
    N, C, S, G = 3, 64, 16384, 8  # L = 131072, 24 segments, forced
    x, g, b = inputs(N, C, S, seed=76)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, f64=True)
    old = ng.norm_get_option(ng.NORM_OPT_BARRIER_TIMEOUT_NS)
    xb, gb, bb = Guarded(N * C * S, x), Guarded(C, g), Guarded(C, b)
    timeouts = 0
    for _ in range(3):
        yb = Guarded(N * C * S)
        ng.norm_set_option(ng.NORM_OPT_GN_PATH, PERS)
        ng.norm_set_option(ng.NORM_OPT_BARRIER_TIMEOUT_NS, 1)
        try:
            ng.norm_group_lrelu_x2_nchw_fwd(xb.t, gb.t, bb.t, yb.t, N, C, S, G, 1e-5, 0.01)
            status = ng.norm_last_error()
        finally:
            ng.norm_set_option(ng.NORM_OPT_BARRIER_TIMEOUT_NS, old)
            ng.norm_set_option(ng.NORM_OPT_GN_PATH, 0)
        assert status in (ng.NORM_OK, ng.NORM_ERR_TIMEOUT)
        timeouts += status == ng.NORM_ERR_TIMEOUT
        got = yb.numpy().astype(np.float64)
        untouched = np.isnan(got)  # the guard sentinel is a NaN no kernel writes
        ok = np.abs(got - want) <= 1e-4 * (1.0 + np.abs(want))
        assert np.all(untouched | ok), "an element of y is neither untouched nor correct"
        assert yb.guards_intact()
    assert timeouts > 0, "a 1 ns limit must make some wait give up"
    assert_parity(run(ng, x, g, b, N, C, S, G, path=PERS), want, "GN NCHW persistent after a timeout")


# ------------------------------------------------------------------ warp path

@pytest.mark.parametrize("N,C,S,G", [(3, 9, 5, 3), (4, 6, 1, 2), (2, 16, 64, 4), (5, 3, 301, 1)])
def test_warp(ng, N, C, S, G):
    check(ng, N, C, S, G, seed=C * S, path=WARP)


# ------------------------------------------------------------------ affine, in place, alignment

@pytest.mark.parametrize("N,C,S,G", [(4, 64, 64, 8), (2, 32, 4096, 4), (3, 9, 5, 3), (1, 8, 1001, 2)])
def test_no_affine_in_place_and_misaligned(ng, N, C, S, G):
    x, _, _ = inputs(N, C, S, seed=41, affine=False)
    want = oracle.group_lrelu_x2_nchw(x, None, None, N, C, S, G, f64=True)
    assert_parity(run(ng, x, None, None, N, C, S, G), want, "GN NCHW no affine")
    assert_parity(run(ng, x, None, None, N, C, S, G, inplace=True), want, "GN NCHW in place")
    x, g, b = inputs(N, C, S, seed=42)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, f64=True)
    assert_parity(run(ng, x, g, b, N, C, S, G, offset=1), want, "GN NCHW misaligned")
    assert_parity(run(ng, x, g, b, N, C, S, G, offset=1, inplace=True), want, "GN NCHW misaligned in place")


@pytest.mark.parametrize("path,cluster", [(REG, 1), (REG, 4), (STREAM, 1), (STREAM, 4), (SPLIT, 0), (WARP, 0),
                                          (PERS, 0)])
def test_in_place_every_path(ng, path, cluster):
    N, C, S, G = 3, 32, 512, 4
    x, g, b = inputs(N, C, S, seed=43)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, f64=True)
    assert_parity(run(ng, x, g, b, N, C, S, G, path=path, cluster=cluster, inplace=True), want,
                  f"GN NCHW in place path={path}")


@pytest.mark.parametrize("slope", [0.0, 0.2, 1.0, -0.5])
def test_slopes(ng, slope):
    check(ng, 2, 64, 256, 16, seed=44, slope=slope)


@pytest.mark.parametrize("path,cluster", [(REG, 0), (REG, 16), (STREAM, 0), (STREAM, 8), (SPLIT, 0), (WARP, 0),
                                          (PERS, 0)])
def test_cancellation(ng, path, cluster):
    # x ~ N(1000, 0.01^2): the mean is 1e5 standard deviations from zero
    N, C, S, G = 2, 16, 4096, 2
    x, g, b = inputs(N, C, S, seed=45, mean=1000.0, std=0.01)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, f64=True)
    assert_parity(run(ng, x, g, b, N, C, S, G, path=path, cluster=cluster), want,
                  f"GN NCHW N(1000, 0.01^2) path={path}")


def test_s1_matches_the_2d_operation(ng):
    N, C, G = 7, 384, 8
    x, g, b = inputs(N, C, 1, seed=46)
    want = oracle.group_lrelu_x2(x, g, b, N, C, G, f64=True)
    assert_parity(run(ng, x, g, b, N, C, 1, G), want, "GN NCHW S = 1")


def test_forced_paths_that_cannot_serve_refuse(ng):
    N, C, S, G = 1, 128, 65536, 32  # L = 262144: no register kernel holds it
    x, g, b = inputs(N, C, S, seed=47)
    with pytest.raises(ng.NormError) as e:
        run(ng, x, g, b, N, C, S, G, path=REG)
    assert e.value.status == ng.NORM_ERR_UNSUPPORTED
    x, g, b = inputs(2, 16, 64, seed=47)
    with pytest.raises(ng.NormError) as e:
        run(ng, x, g, b, 2, 16, 64, 4, path=REG, cluster=2, offset=1)  # not 16-byte aligned
    assert e.value.status == ng.NORM_ERR_UNSUPPORTED
    with pytest.raises(ng.NormError) as e:
        run(ng, x, g, b, 2, 16, 64, 4, path=STREAM, offset=1)
    assert e.value.status == ng.NORM_ERR_UNSUPPORTED
    x, g, b = inputs(1, 8, 4096, seed=47)  # L = 32768: a cluster of 2 cannot hold it
    with pytest.raises(ng.NormError) as e:
        run(ng, x, g, b, 1, 8, 4096, 1, path=REG, cluster=2)
    assert e.value.status == ng.NORM_ERR_UNSUPPORTED


def test_2d_entry_refuses_the_split_path(ng):
    import torch
    x = torch.zeros(64, device="cuda")
    ng.norm_set_option(ng.NORM_OPT_GN_PATH, SPLIT)
    try:
        with pytest.raises(ng.NormError) as e:
            ng.norm_group_lrelu_x2_fwd(x, None, None, x, 4, 16, 4, 1e-5, 0.01)
        assert e.value.status == ng.NORM_ERR_UNSUPPORTED
    finally:
        ng.norm_set_option(ng.NORM_OPT_GN_PATH, 0)


def test_tensor_convenience_4d(ng):
    import torch
    x, g, b = inputs(2, 32, 48, seed=48)
    xt = torch.from_numpy(x).cuda().reshape(2, 32, 6, 8)
    y = ng.group_norm_lrelu_x2(xt, 4, torch.from_numpy(g).cuda(), torch.from_numpy(b).cuda())
    want = oracle.group_lrelu_x2_nchw(x, g, b, 2, 32, 48, 4, f64=True)
    assert_parity(y.cpu().numpy().reshape(-1), want, "group_norm_lrelu_x2 on (2, 32, 6, 8)")
