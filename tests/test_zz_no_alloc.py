"""The allocation-free LayerNorm entry point, norm_layer_fwd_noalloc.

Some callers cannot allocate device memory when they call in: an allocator's
own callbacks, code running under a fixed memory pool, or a plugin that is
handed only its input and output buffers.  This entry point serves them from a
fixed 1 MiB scratch array inside the library instead of a workspace.

Checked here through the C ABI, against the float64 oracle element by element,
on two calls in a row with different inputs (the second call finds the scratch
array as the first left it):
- a shape served by the persistent kernel (tagged records in the array);
- shapes served by the two-kernel path (per-chunk partials in the array): an
  odd row length, and a row length that is a multiple of 4 with that path
  forced;
- a shape served by the row kernel with more rows than the two-kernel path
  could hold partials for (no scratch used, so it is served);
and the persistent shape right after a two-kernel call, so its records start
from an array that holds another path's partials.  A shape whose path needs
more scratch than the array holds is refused before anything is launched.

This file is collected last so that a run stopping at the first failure has
run every other test; it passes alone in a fresh process as well.
"""
import pytest
import torch

import normgen
import oracle
from gpu_util import TOL, Guarded, assert_parity

pytestmark = pytest.mark.gpu

PERSISTENT, SPLIT = 1, 2


@pytest.fixture(scope="module")
def ng():
    import memory_bound_normalization_norm_gb300 as m
    yield m
    m.norm_set_option(m.NORM_OPT_LN_PATH, 0)


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _call_and_check(ng, rows, L, seed, what):
    raw = ng.raw()
    x = normgen.normal(rows * L, 0.5, 2.0, seed=seed, tensor_id=0)
    g = normgen.normal(L, 1.0, 0.1, seed=seed, tensor_id=1)
    b = normgen.normal(L, 0.0, 0.1, seed=seed, tensor_id=2)
    xb, gb, bb = Guarded(rows * L, x), Guarded(L, g), Guarded(L, b)
    yb = Guarded(rows * L)
    st = raw.norm_layer_fwd_noalloc(xb.t.data_ptr(), gb.t.data_ptr(), bb.t.data_ptr(), yb.t.data_ptr(), rows, L,
                                    1e-5, _stream())
    assert st == ng.NORM_OK, ng.norm_status_string(st)
    assert ng.norm_last_error() == ng.NORM_OK
    assert_parity(yb.numpy(), oracle.layer_norm(x, g, b, rows, L, 1e-5), what, TOL)
    assert yb.guards_intact()


@pytest.mark.parametrize("rows,L,path", [
    (3, 1 << 20, 0),          # persistent kernel (automatic choice)
    (5, 7907, 0),             # odd length: two-kernel path
    (9, 152 * 4 * 13, SPLIT),  # two-kernel path forced on a vector shape
    (70000, 8, 0),            # row kernel: no scratch, more rows than the split path could hold
])
def test_noalloc_matches_the_oracle_on_two_calls(ng, rows, L, path):
    ng.norm_set_option(ng.NORM_OPT_LN_PATH, path)
    try:
        for call, seed in enumerate((101, 202)):
            _call_and_check(ng, rows, L, seed, f"no-alloc call {call + 1} {rows}x{L} path {path}")
    finally:
        ng.norm_set_option(ng.NORM_OPT_LN_PATH, 0)


def test_noalloc_persistent_after_split_partials(ng):
    """The two-kernel path leaves arbitrary partials in the array; the persistent
    kernel's tagged records that follow must start from zeros."""
    _call_and_check(ng, 64, 7907, 7, "no-alloc split call")
    _call_and_check(ng, 4, 1 << 20, 8, "no-alloc persistent call after a split call")


def test_noalloc_refuses_shapes_beyond_its_scratch(ng):
    raw = ng.raw()
    rows, L = 70000, 7  # odd length: the two-kernel path, 16 bytes of partials per row > 1 MiB
    assert ng.norm_layer_workspace_bytes(rows, L) > (1 << 20)
    xb, yb = Guarded(rows * L, normgen.normal(rows * L, seed=3)), Guarded(rows * L)
    st = raw.norm_layer_fwd_noalloc(xb.t.data_ptr(), None, None, yb.t.data_ptr(), rows, L, 1e-5, _stream())
    assert st == ng.NORM_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((yb.buf.view(torch.int32) == 0x7FC0DEAD).all()), "a refused call must not write y"
