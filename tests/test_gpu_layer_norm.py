"""LayerNorm on the GPU against the float64 oracle, element by element.

All four paths are covered: the persistent single-read kernel (forced, and chosen
automatically for long rows, over the whole grid or split into row groups), the one-launch row kernel (forced, and chosen
automatically for rows of at most 8,192 elements), the thread-block cluster kernel
shared with GroupNorm (forced, and chosen for fp32 rows of 16,385 to 131,072 over less
than 96 MiB, and for rows of 16,385 to 32,767 over any size) and the
two-kernel split path (forced, and taken for ragged or misaligned rows).  Shapes span several CTAs per row with ragged slices,
rows shorter than one float4 per CTA, the largest row the persistent kernel
holds on chip, and the two full-size workloads: (16, 64, 256, 256) with N(0,1)
inputs and the cancellation stress x ~ N(1000, 0.01^2).
"""
import numpy as np
import pytest
import torch

import normgen
import oracle
from gpu_util import TOL, Guarded, assert_parity, device

pytestmark = pytest.mark.gpu

AUTO, PERSISTENT, SPLIT, ROWS = 0, 1, 2, 3


@pytest.fixture(scope="module")
def ng():
    import memory_bound_normalization_norm_gb300 as m
    yield m
    m.norm_set_option(m.NORM_OPT_LN_PATH, AUTO)


def run_ln(ng, x, g, b, rows, L, eps=1e-5, path=AUTO, offset=0, inplace=False, workspace=None):
    ng.norm_set_option(ng.NORM_OPT_LN_PATH, path)
    xb = Guarded(rows * L, x, offset=offset)
    gd = None if g is None else Guarded(L, g, offset=offset).t
    bd = None if b is None else Guarded(L, b, offset=offset).t
    yb = xb if inplace else Guarded(rows * L, offset=offset)
    if workspace is None:
        ng.norm_layer_fwd(xb.t, gd, bd, yb.t, rows, L, eps)
    else:
        ws, nbytes = workspace
        ng.norm_layer_fwd(xb.t, gd, bd, yb.t, rows, L, eps, ws, nbytes)
    assert ng.norm_last_error() == 0
    ng.norm_set_option(ng.NORM_OPT_LN_PATH, AUTO)
    assert yb.guards_intact(), "LayerNorm wrote outside its output"
    return yb.numpy()


def inputs(rows, L, seed, mean=0.0, std=1.0, affine=True):
    x = normgen.normal(rows * L, mean, std, seed=seed, tensor_id=0)
    if not affine:
        return x, None, None
    g = normgen.normal(L, 1.0, 0.1, seed=seed, tensor_id=1)
    b = normgen.normal(L, 0.0, 0.1, seed=seed, tensor_id=2)
    return x, g, b


SHAPES = [
    (1, 4), (2, 64), (3, 600), (5, 4 * 152 * 13 + 4), (2, 65536 + 4), (4, 1 << 18), (1, 3 * (1 << 20)),
]


@pytest.mark.parametrize("path", [PERSISTENT, SPLIT])
@pytest.mark.parametrize("rows,L", SHAPES)
def test_layer_norm_paths(ng, path, rows, L):
    x, g, b = inputs(rows, L, seed=rows * 7 + L)
    want = oracle.layer_norm(x, g, b, rows, L)
    assert_parity(run_ln(ng, x, g, b, rows, L, path=path), want, f"LN path={path} {rows}x{L}")


@pytest.mark.parametrize("rows,L", [(1, 1), (2, 3), (3, 1001), (4, 4097), (2, 100003)])
def test_layer_norm_ragged_rows(ng, rows, L):
    x, g, b = inputs(rows, L, seed=L)
    assert_parity(run_ln(ng, x, g, b, rows, L), oracle.layer_norm(x, g, b, rows, L), f"LN ragged {rows}x{L}")


@pytest.mark.parametrize("path", [AUTO, SPLIT])
def test_layer_norm_misaligned_pointers(ng, path):
    rows, L = 3, 8192
    x, g, b = inputs(rows, L, seed=11)
    got = run_ln(ng, x, g, b, rows, L, path=path, offset=1)
    assert_parity(got, oracle.layer_norm(x, g, b, rows, L), "LN misaligned")


@pytest.mark.parametrize("path", [PERSISTENT, SPLIT])
def test_layer_norm_identity_affine_and_in_place(ng, path):
    rows, L = 3, 152 * 4 * 20
    x, _, _ = inputs(rows, L, seed=5, affine=False)
    want = oracle.layer_norm(x, None, None, rows, L)
    assert_parity(run_ln(ng, x, None, None, rows, L, path=path), want, "LN no affine")
    assert_parity(run_ln(ng, x, None, None, rows, L, path=path, inplace=True), want, "LN in place")


@pytest.mark.parametrize("path", [PERSISTENT, SPLIT])
def test_layer_norm_constant_rows_give_beta(ng, path):
    rows, L = 2, 152 * 4 * 3
    x = np.full(rows * L, 3.5, dtype=np.float32)
    _, g, b = inputs(rows, L, seed=9)
    got = run_ln(ng, x, g, b, rows, L, path=path).reshape(rows, L)
    assert np.array_equal(got, np.stack([b, b])), "constant row must give exactly beta"


def test_layer_norm_largest_resident_row(ng):
    L = ng.norm_layer_max_resident_row_len()
    assert L >= 64 * 256 * 256, "the (64, 256, 256) row must fit on chip"
    x, g, b = inputs(2, L, seed=3)
    got = run_ln(ng, x, g, b, 2, L, path=PERSISTENT)
    assert_parity(got, oracle.layer_norm(x, g, b, 2, L), "LN largest resident row")
    with pytest.raises(ng.NormError):
        ng.norm_set_option(ng.NORM_OPT_LN_PATH, PERSISTENT)
        try:
            xd = torch.zeros(L + 4, device="cuda")
            ng.norm_layer_fwd(xd, None, None, xd, 1, L + 4, 1e-5)
        finally:
            ng.norm_set_option(ng.NORM_OPT_LN_PATH, AUTO)


def test_layer_norm_caller_workspace_reused(ng):
    rows, L = 4, 152 * 4 * 50
    nbytes = ng.norm_layer_workspace_bytes(rows, L)
    ws = torch.zeros((nbytes + 255) // 4 + 64, dtype=torch.float32, device="cuda")
    for seed in (1, 2, 3):
        for path in (PERSISTENT, SPLIT):
            x, g, b = inputs(rows, L, seed=seed)
            got = run_ln(ng, x, g, b, rows, L, path=path, workspace=(ws, nbytes))
            assert_parity(got, oracle.layer_norm(x, g, b, rows, L), f"LN caller workspace seed={seed}")
    # a shape the two-kernel path serves needs more than 16 bytes of workspace
    small = torch.zeros(1 << 18, dtype=torch.float32, device="cuda")
    with pytest.raises(ng.NormError) as e:
        ng.norm_layer_fwd(small, None, None, small, 1, 1 << 18, 1e-5, ws, 16)
    assert e.value.status == ng.NORM_ERR_WORKSPACE


def test_layer_norm_deterministic(ng):
    rows, L = 3, 1 << 20
    x, g, b = inputs(rows, L, seed=21)
    a = run_ln(ng, x, g, b, rows, L, path=PERSISTENT)
    c = run_ln(ng, x, g, b, rows, L, path=PERSISTENT)
    assert a.tobytes() == c.tobytes()


def test_persistent_exchange_200_launches_back_to_back(ng):
    """The grid exchange across 200 persistent launches queued back to back on one
    stream and one caller workspace, with no synchronization between them.  The
    inputs cycle through 8 seeded tensors of different means and spreads, so a
    record read from the wrong row, the wrong slot or the previous launch (a stale
    or torn word accepted by its tag) would give visibly wrong statistics.  Each
    launch writes its own output; every element of every output is compared with
    the oracle.  6 rows a launch cycle the 4 record slots 300 times and the tags
    through 1,200 rows."""
    rows, L, launches, distinct = 6, 1 << 20, 200, 8
    sets, wants = [], []
    for k in range(distinct):
        x, g, b = inputs(rows, L, seed=500 + k, mean=3.0 * k - 10.0, std=0.5 + k)
        sets.append((device(x), device(g), device(b)))
        wants.append(oracle.layer_norm(x, g, b, rows, L))
    nbytes = ng.norm_layer_workspace_bytes(rows, L)
    ws = torch.zeros((nbytes + 255) // 4 + 64, dtype=torch.float32, device="cuda")
    ys = torch.full((launches, rows * L), float("nan"), dtype=torch.float32, device="cuda")
    ng.norm_set_option(ng.NORM_OPT_LN_PATH, PERSISTENT)
    try:
        for i in range(launches):
            xd, gd, bd = sets[i % distinct]
            ng.norm_layer_fwd(xd, gd, bd, ys[i], rows, L, 1e-5, ws, nbytes)
    finally:
        ng.norm_set_option(ng.NORM_OPT_LN_PATH, AUTO)
    assert ng.norm_last_error() == 0
    for k in range(distinct):
        want = torch.from_numpy(wants[k].astype(np.float64)).cuda()
        got = ys[k::distinct].double()
        err = ((got - want).abs() / (1.0 + want.abs())).amax(dim=1)
        assert bool(torch.isfinite(got).all()), f"input {k}: a launch left NaN in its output"
        worst = float(err.max())
        assert worst <= TOL, f"input {k}: worst launch {int(err.argmax()) * distinct + k} scaled error {worst:.3e}"


@pytest.mark.parametrize("rows,L,path", [
    (256, 262144, AUTO),        # 15 row groups of 10 CTAs (the automatic choice)
    (64, 1 << 20, AUTO),        # 4 groups of 38
    (11, (1 << 20) + 4, AUTO),  # 4 groups, 3, 3, 3 and 2 rows
    (3, 1 << 20, AUTO),         # one row per group
    (40, 131076, PERSISTENT),   # 30 groups of 5 CTAs, forced
    (7, 200004, PERSISTENT),    # a length that is not a multiple of the group size (5.6 MB: forced)
    (1024, 32768, AUTO),        # 128 MiB of rows of 32,768: 76 groups of 2 CTAs (automatic)
    (384, 65536, AUTO),         # 96 MiB of rows of 65,536: 50 groups of 3 CTAs (automatic)
])
def test_persistent_row_groups(ng, rows, L, path):
    """Rows of 131,073 to about 1.6 Mi elements, and rows of 32,768 or more over 96 MiB:
    the persistent kernel splits its grid into row groups, each taking every k-th row
    with its own grid exchange."""
    x, g, b = inputs(rows, L, seed=rows + L)
    want = oracle.layer_norm(x, g, b, rows, L)
    assert_parity(run_ln(ng, x, g, b, rows, L, path=path), want, f"LN row groups {rows}x{L}")
    # the cancellation stress through the same groups
    xs = normgen.normal(rows * L, 1000.0, 1e-2, seed=rows, tensor_id=0)
    ws = oracle.layer_norm(xs, None, None, rows, L)
    assert_parity(run_ln(ng, xs, None, None, rows, L, path=path), ws, f"LN row groups stress {rows}x{L}")


def test_layer_norm_empty_is_noop(ng):
    yb = Guarded(16)
    ng.norm_layer_fwd(None, None, None, yb.t, 0, 16, 1e-5)
    ng.norm_layer_fwd(yb.t, None, None, yb.t, 4, 0, 1e-5)
    torch.cuda.synchronize()
    assert (yb.buf.view(torch.int32) == 0x7FC0DEAD).all()


@pytest.mark.slow
@pytest.mark.parametrize("path", [AUTO, SPLIT])
def test_layer_norm_full_size_normal(ng, path):
    """(16, 64, 256, 256) over the last 3 dims, x ~ N(0,1), gamma ~ N(1,0.1), beta ~ N(0,0.1)."""
    rows, L = 16, 64 * 256 * 256
    x, g, b = inputs(rows, L, seed=0)
    want = oracle.layer_norm(x, g, b, rows, L)
    assert_parity(run_ln(ng, x, g, b, rows, L, path=path), want, f"LN full size path={path}")


@pytest.mark.slow
@pytest.mark.parametrize("path", [AUTO, SPLIT])
def test_layer_norm_full_size_cancellation_stress(ng, path):
    """(16, 64, 256, 256), x ~ N(1000, 0.01^2), gamma = 1, beta = 0 passed as tensors."""
    rows, L = 16, 64 * 256 * 256
    x = normgen.normal(rows * L, 1000.0, 1e-2, seed=0, tensor_id=0)
    g = np.ones(L, dtype=np.float32)
    b = np.zeros(L, dtype=np.float32)
    want = oracle.layer_norm(x, g, b, rows, L)
    err = assert_parity(run_ln(ng, x, g, b, rows, L, path=path), want, f"LN stress path={path}")
    assert err < TOL / 4, f"cancellation stress margin too thin: {err:.2e}"


ROW_SHAPES = [(1, 4), (3, 12), (7, 1000), (256, 1024), (64, 4096), (33, 8192), (9, 16384), (2, 16380),
              (3000, 64)]


@pytest.mark.parametrize("rows,L", ROW_SHAPES)
def test_layer_norm_row_kernel(ng, rows, L):
    x, g, b = inputs(rows, L, seed=rows + 3 * L)
    want = oracle.layer_norm(x, g, b, rows, L)
    forced = run_ln(ng, x, g, b, rows, L, path=ROWS)
    assert_parity(forced, want, f"LN row kernel {rows}x{L}")
    if L <= 8192:
        # chosen automatically for these shapes: the same bits
        assert np.array_equal(run_ln(ng, x, g, b, rows, L), forced)
    else:
        assert_parity(run_ln(ng, x, g, b, rows, L), want, f"LN auto {rows}x{L}")


def test_layer_norm_row_kernel_stress_in_place_and_no_affine(ng):
    rows, L = 8, 16384
    x, _, _ = inputs(rows, L, seed=77, mean=1000.0, std=1e-2, affine=False)
    ones, zeros = np.ones(L, np.float32), np.zeros(L, np.float32)
    want = oracle.layer_norm(x, ones, zeros, rows, L)
    assert_parity(run_ln(ng, x, ones, zeros, rows, L, path=ROWS), want, "LN row kernel stress")
    assert_parity(run_ln(ng, x, None, None, rows, L, path=ROWS), want, "LN row kernel no affine")
    assert_parity(run_ln(ng, x, None, None, rows, L, path=ROWS, inplace=True), want, "LN row kernel in place")


@pytest.mark.parametrize("L,offset", [(16388, 0), (1002, 0), (1024, 1)])
def test_layer_norm_row_kernel_refuses_what_it_cannot_take(ng, L, offset):
    # longer than 16,384, not a multiple of 4, or misaligned: forced, it refuses;
    # automatically, another path serves the shape
    rows = 2
    x, g, b = inputs(rows, L, seed=L)
    ng.norm_set_option(ng.NORM_OPT_LN_PATH, ROWS)
    try:
        xb, yb = Guarded(rows * L, x, offset=offset), Guarded(rows * L, offset=offset)
        with pytest.raises(ng.NormError) as e:
            ng.norm_layer_fwd(xb.t, None, None, yb.t, rows, L, 1e-5)
        assert e.value.status == ng.NORM_ERR_UNSUPPORTED
    finally:
        ng.norm_set_option(ng.NORM_OPT_LN_PATH, AUTO)
    assert_parity(run_ln(ng, x, g, b, rows, L, offset=offset), oracle.layer_norm(x, g, b, rows, L),
                  f"LN auto {rows}x{L}")


@pytest.mark.parametrize("rows,L,offset", [(24, 1 << 19, 0), (11, (1 << 20) + 1, 1)])
def test_split_path_large(ng, rows, L, offset):
    # 50 MB of x through the two-kernel path: vector form, and scalar form with a
    # ragged length and misaligned pointers
    x, g, b = inputs(rows, L, seed=rows + L)
    want = oracle.layer_norm(x, g, b, rows, L)
    assert_parity(run_ln(ng, x, g, b, rows, L, path=SPLIT, offset=offset), want, f"LN large split {rows}x{L}")
    assert_parity(run_ln(ng, x, g, b, rows, L, path=SPLIT, offset=offset, inplace=True), want,
                  f"LN large split in place {rows}x{L}")


STREAM = 4


@pytest.mark.parametrize("rows,L", [(3, 4096), (5, 20000), (2, 131072), (7, 65544), (300, 2048), (33, 16388)])
def test_streamed_cluster_kernel(ng, rows, L):
    # the cluster kernel shared with GroupNorm: one CTA (L <= 8192) or a cluster
    # of up to 16 per row, slices by bulk copy, one exchange of partials per row
    x, g, b = inputs(rows, L, seed=rows + 3 * L)
    want = oracle.layer_norm(x, g, b, rows, L)
    assert_parity(run_ln(ng, x, g, b, rows, L, path=STREAM), want, f"LN streamed {rows}x{L}")
    assert_parity(run_ln(ng, x, g, b, rows, L, path=STREAM, inplace=True), want, f"LN streamed in place {rows}x{L}")
    xn, _, _ = inputs(rows, L, seed=rows + 3 * L, affine=False)
    assert_parity(run_ln(ng, xn, None, None, rows, L, path=STREAM), oracle.layer_norm(xn, None, None, rows, L),
                  f"LN streamed no affine {rows}x{L}")


def test_streamed_cluster_kernel_cancellation(ng):
    rows, L = 6, 65536
    x, _, _ = inputs(rows, L, seed=77, mean=1000.0, std=0.01, affine=False)
    assert_parity(run_ln(ng, x, None, None, rows, L, path=STREAM), oracle.layer_norm(x, None, None, rows, L),
                  "LN streamed N(1000, 0.01^2)")


def test_streamed_cluster_kernel_refusals(ng):
    x, g, b = inputs(2, 4096, seed=78)
    with pytest.raises(ng.NormError) as e:
        run_ln(ng, x, g, b, 2, 4096, path=STREAM, offset=1)  # not 16-byte aligned
    assert e.value.status == ng.NORM_ERR_UNSUPPORTED
    x, g, b = inputs(1, 262144, seed=79)
    with pytest.raises(ng.NormError) as e:
        run_ln(ng, x, g, b, 1, 262144, path=STREAM)  # longer than 16 CTAs hold
    assert e.value.status == ng.NORM_ERR_UNSUPPORTED
    ng.norm_set_option(ng.NORM_OPT_LN_PATH, AUTO)
