"""Failure detection of the LayerNorm grid barrier, without faulting the GPU.

The persistent kernel's grid barrier is told to wait for one arrival more than
there are CTAs, so it can only end by running out its (2 ms) limit.  Every CTA
must then record NORM_ERR_TIMEOUT, drain its own bulk copies and return without
writing y; norm_last_error() reports the status and resets the library-owned
workspace, after which a normal call works again.
"""
import pytest
import torch

import normgen
import oracle
from gpu_util import Guarded, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture()
def ng():
    import memory_bound_normalization_norm_gb300 as m
    yield m
    m.norm_set_option(m.NORM_OPT_BARRIER_EXTRA_ARRIVALS, 0)
    m.norm_set_option(m.NORM_OPT_BARRIER_TIMEOUT_NS, 200_000_000)
    m.norm_set_option(m.NORM_OPT_LN_PATH, 0)


def test_barrier_timeout_is_reported_and_recoverable(ng):
    rows, L = 3, 152 * 4 * 64
    x = normgen.normal(rows * L, seed=1)
    xb = Guarded(rows * L, x)
    yb = Guarded(rows * L)
    assert ng.norm_last_error() == 0
    ng.norm_set_option(ng.NORM_OPT_LN_PATH, 1)
    ng.norm_set_option(ng.NORM_OPT_BARRIER_TIMEOUT_NS, 2_000_000)
    ng.norm_set_option(ng.NORM_OPT_BARRIER_EXTRA_ARRIVALS, 1)
    ng.norm_layer_fwd(xb.t, None, None, yb.t, rows, L, 1e-5)
    assert ng.norm_last_error() == ng.NORM_ERR_TIMEOUT
    assert ng.norm_last_error() == 0, "the error word must be cleared once read"
    bits = yb.buf.view(torch.int32)
    assert bool((bits == 0x7FC0DEAD).all()), "a timed-out call must not write y"

    ng.norm_set_option(ng.NORM_OPT_BARRIER_EXTRA_ARRIVALS, 0)
    ng.norm_set_option(ng.NORM_OPT_BARRIER_TIMEOUT_NS, 200_000_000)
    ng.norm_layer_fwd(xb.t, None, None, yb.t, rows, L, 1e-5)
    assert ng.norm_last_error() == 0
    assert_parity(yb.numpy(), oracle.layer_norm(x, None, None, rows, L), "LN after recovery")
    assert yb.guards_intact()
