"""Failure detection of the persistent LayerNorm kernel, without faulting the GPU.

1. The grid barrier is told to wait for records no CTA publishes, so it can only
   end by running out its (2 ms) limit.  Every CTA must record NORM_ERR_TIMEOUT,
   drain its own bulk copies and return without writing y; norm_last_error()
   reports the status and resets the library-owned workspace, after which a
   normal call works again.
2. A 1 ns limit makes the other waits give up too (a row's bulk copy that has
   not landed at the first, non-blocking look, as row 0 has not at the start):
   the CTA still records the error and drains its copies; every element of y
   is then either untouched or correct.
3. Error words are per stream: a timeout on one stream is reported by
   norm_last_error on that stream only.
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


@pytest.mark.parametrize("rows", [3, 1])  # three row groups; one group (the one-group form)
def test_barrier_timeout_is_reported_and_recoverable(ng, rows):
    L = 152 * 4 * 64
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


@pytest.mark.parametrize("rows", [3, 1])  # three row groups; one group (the one-group form)
def test_tiny_wait_limit_aborts_cleanly(ng, rows):
    """A 1 ns limit makes any wait that is not over at its first look give up: the
    statistics and apply warps' waits for a row's bulk copy (row 0 has not landed
    when they first look), or warp 0's poll.  Whichever gives up, the CTA must record
    NORM_ERR_TIMEOUT and drain its copies (drains wait at least 100 ms whatever the
    limit).  CTAs stop independently, so y may be partly written: every element is
    untouched or correct.  Then a normal call works."""
    L = 152 * 4 * 64
    x, g, b = (normgen.normal(rows * L, seed=5), normgen.normal(L, 1.0, 0.1, seed=5, tensor_id=1),
               normgen.normal(L, 0.0, 0.1, seed=5, tensor_id=2))
    want = oracle.layer_norm(x, g, b, rows, L).reshape(rows, L)
    xb, gb, bb = Guarded(rows * L, x), Guarded(L, g), Guarded(L, b)
    assert ng.norm_last_error() == 0
    ng.norm_set_option(ng.NORM_OPT_LN_PATH, 1)
    timeouts = 0
    for _ in range(3):
        yb = Guarded(rows * L)
        ng.norm_set_option(ng.NORM_OPT_BARRIER_TIMEOUT_NS, 1)
        ng.norm_layer_fwd(xb.t, gb.t, bb.t, yb.t, rows, L, 1e-5)
        st = ng.norm_last_error()
        ng.norm_set_option(ng.NORM_OPT_BARRIER_TIMEOUT_NS, 200_000_000)
        assert st in (ng.NORM_OK, ng.NORM_ERR_TIMEOUT)
        timeouts += st == ng.NORM_ERR_TIMEOUT
        got = yb.numpy().reshape(rows, L)
        written = (yb.t.view(torch.int32).reshape(rows, L) != 0x7FC0DEAD).cpu().numpy()
        if st == ng.NORM_OK:
            assert written.all()
        # CTAs vote to stop independently, so a row may be written by some CTAs
        # and not others: every element is untouched or correct
        assert_parity(got[written], want[written], f"written elements after a 1 ns limit (status {st})")
        assert yb.guards_intact()
    assert timeouts > 0, "a 1 ns limit must make some wait give up"
    yb = Guarded(rows * L)
    ng.norm_layer_fwd(xb.t, gb.t, bb.t, yb.t, rows, L, 1e-5)
    assert ng.norm_last_error() == 0
    assert_parity(yb.numpy(), want.reshape(-1), "LN after the aborted calls")


def test_error_word_is_per_stream(ng):
    rows, L = 3, 152 * 4 * 64
    xb, yb = Guarded(rows * L, normgen.normal(rows * L, seed=9)), Guarded(rows * L)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    assert ng.norm_last_error(sa) == 0 and ng.norm_last_error(sb) == 0
    ng.norm_set_option(ng.NORM_OPT_LN_PATH, 1)
    ng.norm_set_option(ng.NORM_OPT_BARRIER_TIMEOUT_NS, 2_000_000)
    ng.norm_set_option(ng.NORM_OPT_BARRIER_EXTRA_ARRIVALS, 1)
    torch.cuda.synchronize()
    ng.norm_layer_fwd(xb.t, None, None, yb.t, rows, L, 1e-5, stream=sa)
    ng.norm_set_option(ng.NORM_OPT_BARRIER_EXTRA_ARRIVALS, 0)
    ng.norm_set_option(ng.NORM_OPT_BARRIER_TIMEOUT_NS, 200_000_000)
    sa.synchronize()
    assert ng.norm_last_error(sb) == 0, "a timeout on another stream must not be reported here"
    assert ng.norm_last_error() == 0, "nor on the current stream"
    assert ng.norm_last_error(sa) == ng.NORM_ERR_TIMEOUT
    assert ng.norm_last_error(sa) == 0
