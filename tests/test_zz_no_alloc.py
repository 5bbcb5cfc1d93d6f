"""The allocation-free LayerNorm entry point, norm_layer_fwd_noalloc.

Some callers cannot allocate device memory when they call in: an allocator's
own callbacks, code running under a fixed memory pool, or a plugin that is
handed only its input and output buffers.  This entry point serves them from a
fixed 1 MiB scratch array inside the library instead of a workspace.

Checked here through the C ABI: its output matches norm_layer_fwd's within the
parity tolerance on two calls in a row (the second call finds the scratch array
as the first left it), for a shape served by the persistent kernel and one
served by the two-kernel path; and a shape that needs more scratch than the
array holds is refused before anything is launched.

This file is collected last so that a run stopping at the first failure has
run every other test; it passes alone in a fresh process as well.
"""
import pytest
import torch

import normgen
from gpu_util import TOL, Guarded, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ng():
    import memory_bound_normalization_norm_gb300 as m
    return m


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("rows,L", [(3, 1 << 20), (5, 152 * 4 * 13 + 4)])
def test_noalloc_matches_norm_layer_fwd_on_two_calls(ng, rows, L):
    raw = ng.raw()
    for call, seed in enumerate((101, 202)):
        x = normgen.normal(rows * L, 0.5, 2.0, seed=seed, tensor_id=0)
        g = normgen.normal(L, 1.0, 0.1, seed=seed, tensor_id=1)
        b = normgen.normal(L, 0.0, 0.1, seed=seed, tensor_id=2)
        xb, gb, bb = Guarded(rows * L, x), Guarded(L, g), Guarded(L, b)
        y_ref, y_new = Guarded(rows * L), Guarded(rows * L)
        st = raw.norm_layer_fwd(xb.t.data_ptr(), gb.t.data_ptr(), bb.t.data_ptr(), y_ref.t.data_ptr(), rows, L,
                                1e-5, None, 0, _stream())
        assert st == ng.NORM_OK
        st = raw.norm_layer_fwd_noalloc(xb.t.data_ptr(), gb.t.data_ptr(), bb.t.data_ptr(), y_new.t.data_ptr(),
                                        rows, L, 1e-5, _stream())
        assert st == ng.NORM_OK, ng.norm_status_string(st)
        assert ng.norm_last_error() == ng.NORM_OK
        assert_parity(y_new.numpy(), y_ref.numpy(), f"no-alloc call {call + 1} {rows}x{L}", TOL)
        assert y_new.guards_intact()


def test_noalloc_refuses_shapes_beyond_its_scratch(ng):
    raw = ng.raw()
    rows, L = 70000, 8  # needs 16 bytes of scratch per row on the two-kernel path: > 1 MiB
    assert ng.norm_layer_workspace_bytes(rows, L) > (1 << 20)
    xb, yb = Guarded(rows * L, normgen.normal(rows * L, seed=3)), Guarded(rows * L)
    st = raw.norm_layer_fwd_noalloc(xb.t.data_ptr(), None, None, yb.t.data_ptr(), rows, L, 1e-5, _stream())
    assert st == ng.NORM_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((yb.buf.view(torch.int32) == 0x7FC0DEAD).all()), "a refused call must not write y"
