"""Channel RMSNorm on the GPU against the float64 oracle, element by element.

Covers every register-resident channel bucket (exact and ragged C up to 128),
the two-read kernel (C > 128), odd spatial sizes, in place, misaligned pointers,
and the small (2, 64, 32, 32) workload in full.  The (112, 64, 512, 512) workload
(7.5 GB in) is compared element by element, one batch entry at a time, in
test_gpu_bench_shapes.py.
"""
import numpy as np
import pytest
import torch

import normgen
import oracle
from gpu_util import Guarded, assert_parity, device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ng():
    import memory_bound_normalization_norm_gb300 as m
    return m


def run_rms(ng, x, B, C, S, eps=1e-5, offset=0, inplace=False):
    xb = Guarded(B * C * S, x, offset=offset)
    yb = xb if inplace else Guarded(B * C * S, offset=offset)
    ng.norm_rms_channel_fwd(xb.t, yb.t, B, C, S, eps)
    out = yb.numpy()
    assert yb.guards_intact(), "RMSNorm wrote outside its output"
    return out


@pytest.mark.parametrize("C", [1, 2, 3, 4, 5, 8, 13, 16, 31, 32, 33, 63, 64, 65, 100, 128, 129, 200])
@pytest.mark.parametrize("B,S", [(1, 1), (3, 257), (2, 4096)])
def test_channels(ng, C, B, S):
    x = normgen.normal(B * C * S, seed=C * 1000 + S, tensor_id=0)
    assert_parity(run_rms(ng, x, B, C, S), oracle.rms_channel(x, B, C, S), f"RMS B={B} C={C} S={S}")


@pytest.mark.parametrize("B,C,S", [(2, 33, 40000), (3, 64, 30000), (1, 17, 70001)])
def test_more_positions_than_one_wave(ng, B, C, S):
    # 30,000 to 80,000 positions: several position blocks per batch entry, with
    # exact and predicated channel counts
    x = normgen.normal(B * C * S, seed=B + C + S, tensor_id=0)
    assert_parity(run_rms(ng, x, B, C, S), oracle.rms_channel(x, B, C, S), f"RMS B={B} C={C} S={S}")


def test_in_place_and_misaligned(ng):
    B, C, S = 3, 64, 1023
    x = normgen.normal(B * C * S, seed=5)
    want = oracle.rms_channel(x, B, C, S)
    assert_parity(run_rms(ng, x, B, C, S, inplace=True), want, "RMS in place")
    assert_parity(run_rms(ng, x, B, C, S, offset=1), want, "RMS misaligned")


def test_zero_input_is_zero(ng):
    B, C, S = 2, 64, 300
    x = np.zeros(B * C * S, dtype=np.float32)
    assert np.array_equal(run_rms(ng, x, B, C, S), x)


def test_large_values_do_not_overflow(ng):
    B, C, S = 1, 64, 512
    x = normgen.normal(B * C * S, 0.0, 1e18, seed=6)
    assert_parity(run_rms(ng, x, B, C, S), oracle.rms_channel(x, B, C, S), "RMS large values")


def test_small_workload_full(ng):
    """(2, 64, 32, 32), x ~ N(0,1) seed 0, eps 1e-5."""
    B, C, S = 2, 64, 32 * 32
    x = normgen.normal(B * C * S, seed=0, tensor_id=0)
    assert_parity(run_rms(ng, x, B, C, S), oracle.rms_channel(x, B, C, S), "RMS (2,64,32,32)")


def test_many_batches_fold_grid(ng):
    B, C, S = 70000, 4, 3
    x = normgen.normal(B * C * S, seed=7)
    assert_parity(run_rms(ng, x, B, C, S), oracle.rms_channel(x, B, C, S), "RMS 70000 batches")
