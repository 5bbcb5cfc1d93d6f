"""Chains of calls on one stream, each reading the output of the call before it, against the oracle.

Consecutive kernels of one stream may overlap under programmatic dependent launch.  The (N, C)
GroupNorm, row LayerNorm and team kernels let the next kernel be scheduled at their start; the
streamed cluster kernel's GroupNorm form does so once its last segment's statistics are merged.
Every kernel launched that way waits for its predecessor's completion, and for its writes to be
visible, before its first global access.  These tests check that each stage of a chain reads the
finished output of the stage before: every stage is compared with the oracle applied to the
GPU's own output of the previous stage, and the intermediate buffers hold NaN before each pass of
the chain, so a stage that read too early would see NaN or a part of the previous pass.
"""
import numpy as np
import pytest
import torch

import normgen
import oracle
from gpu_util import assert_bf16_parity, assert_parity, bf16_device, bf16_values

pytestmark = pytest.mark.gpu

# (8, 512, 64, 64) NCHW with 32 groups: the streamed cluster kernel's GroupNorm form
N4, C4, S4, G4 = 8, 512, 4096, 32
# the same 16,777,216 values as (N, C) rows of 8,192 channels in 512 groups of 16
NR, CR, GR = 2048, 8192, 512
# and as LayerNorm rows of 4,096 (the row kernel)
LR, LL = 4096, 4096
EPS, SLOPE = 1e-5, 0.01


@pytest.fixture(scope="module")
def ng():
    import memory_bound_normalization_norm_gb300 as m
    return m


def params(n, seed):
    g = normgen.normal(n, 1.0, 0.1, seed=seed, tensor_id=1)
    b = normgen.normal(n, 0.0, 0.1, seed=seed, tensor_id=2)
    return g, b


def test_fp32_chain(ng):
    x = normgen.normal(N4 * C4 * S4, seed=71, tensor_id=0)
    gc, bc = params(C4, 72)    # NCHW GroupNorm, per channel
    gr, br = params(CR, 73)    # (N, C) GroupNorm
    gl, bl = params(LL, 74)    # LayerNorm rows
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    xd, gcd, bcd, grd, brd, gld, bld = (dev(a) for a in (x, gc, bc, gr, br, gl, bl))
    y = [torch.empty_like(xd) for _ in range(5)]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(s):
            for t in y:
                t.fill_(float("nan"))
            st = s.cuda_stream
            # (N, C) GroupNorm -> NCHW GroupNorm -> NCHW GroupNorm -> the same in place
            # -> LayerNorm rows -> NCHW GroupNorm, with no synchronization in between
            ng.norm_group_lrelu_x2_fwd(xd, grd, brd, y[0], NR, CR, GR, EPS, SLOPE, stream=st)
            ng.norm_group_lrelu_x2_nchw_fwd(y[0], gcd, bcd, y[1], N4, C4, S4, G4, EPS, SLOPE, stream=st)
            ng.norm_group_lrelu_x2_nchw_fwd(y[1], gcd, bcd, y[2], N4, C4, S4, G4, EPS, SLOPE, stream=st)
            # snapshot of the third stage's output, taken in stream order before it is overwritten
            y2_copy = y[2].clone()
            ng.norm_group_lrelu_x2_nchw_fwd(y[2], gcd, bcd, y[2], N4, C4, S4, G4, EPS, SLOPE, stream=st)
            ng.norm_layer_fwd(y[2], gld, bld, y[3], LR, LL, EPS, stream=st)
            ng.norm_group_lrelu_x2_nchw_fwd(y[3], gcd, bcd, y[4], N4, C4, S4, G4, EPS, SLOPE, stream=st)
        torch.cuda.synchronize()
        assert ng.norm_last_error(s.cuda_stream) == 0
        got = [t.cpu().numpy() for t in y]
        y2_in = y2_copy.cpu().numpy()
        assert_parity(got[0], oracle.group_lrelu_x2(x, gr, br, NR, CR, GR, EPS, SLOPE), "(N, C) GroupNorm")
        assert_parity(got[1], oracle.group_lrelu_x2_nchw(got[0], gc, bc, N4, C4, S4, G4, EPS, SLOPE),
                      "NCHW GroupNorm after (N, C) GroupNorm")
        assert_parity(y2_in, oracle.group_lrelu_x2_nchw(got[1], gc, bc, N4, C4, S4, G4, EPS, SLOPE),
                      "NCHW GroupNorm after NCHW GroupNorm")
        assert_parity(got[2], oracle.group_lrelu_x2_nchw(y2_in, gc, bc, N4, C4, S4, G4, EPS, SLOPE),
                      "NCHW GroupNorm in place after NCHW GroupNorm")
        assert_parity(got[3], oracle.layer_norm(got[2], gl, bl, LR, LL, EPS), "LayerNorm rows after NCHW GroupNorm")
        assert_parity(got[4], oracle.group_lrelu_x2_nchw(got[3], gc, bc, N4, C4, S4, G4, EPS, SLOPE),
                      "NCHW GroupNorm after LayerNorm rows")


def test_bf16_chain(ng):
    x = normgen.normal(N4 * C4 * S4, seed=81, tensor_id=0)
    gc, bc = params(C4, 82)
    gr, br = params(CR, 83)
    # parameters as bf16 values; the oracle takes the same values widened
    xd, gcd, bcd, grd, brd = (bf16_device(a) for a in (x, gc, bc, gr, br))
    x, gc, bc, gr, br = (bf16_values(t) for t in (xd, gcd, bcd, grd, brd))
    y = [torch.empty_like(xd) for _ in range(4)]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(s):
            for t in y:
                t.fill_(float("nan"))
            st = s.cuda_stream
            # NCHW GroupNorm -> NCHW GroupNorm -> (N, C) GroupNorm (8 channels a thread)
            # -> NCHW GroupNorm
            ng.norm_group_lrelu_x2_nchw_fwd_bf16(xd, gcd, bcd, y[0], N4, C4, S4, G4, EPS, SLOPE, stream=st)
            ng.norm_group_lrelu_x2_nchw_fwd_bf16(y[0], gcd, bcd, y[1], N4, C4, S4, G4, EPS, SLOPE, stream=st)
            ng.norm_group_lrelu_x2_fwd_bf16(y[1], grd, brd, y[2], NR, CR, GR, EPS, SLOPE, stream=st)
            ng.norm_group_lrelu_x2_nchw_fwd_bf16(y[2], gcd, bcd, y[3], N4, C4, S4, G4, EPS, SLOPE, stream=st)
        torch.cuda.synchronize()
        assert ng.norm_last_error(s.cuda_stream) == 0
        got = [bf16_values(t) for t in y]
        assert_bf16_parity(got[0], oracle.group_lrelu_x2_nchw(x, gc, bc, N4, C4, S4, G4, EPS, SLOPE),
                           "bf16 NCHW GroupNorm")
        assert_bf16_parity(got[1], oracle.group_lrelu_x2_nchw(got[0], gc, bc, N4, C4, S4, G4, EPS, SLOPE),
                           "bf16 NCHW GroupNorm after NCHW GroupNorm")
        assert_bf16_parity(got[2], oracle.group_lrelu_x2(got[1], gr, br, NR, CR, GR, EPS, SLOPE),
                           "bf16 (N, C) GroupNorm after NCHW GroupNorm")
        assert_bf16_parity(got[3], oracle.group_lrelu_x2_nchw(got[2], gc, bc, N4, C4, S4, G4, EPS, SLOPE),
                           "bf16 NCHW GroupNorm after (N, C) GroupNorm")
