"""The bfloat16 entry points on the GPU against the float64 oracle, element by element.

Inputs are the seeded float32 streams rounded to bfloat16, so the oracle sees exactly
the values the GPU reads.  The GPU computes in fp32 and rounds y to bfloat16 once;
the oracle's float64 result is not rounded.  The bound per element is therefore the
bfloat16 rounding of the result, 2^-8 |y_ref| (half an ulp of 8 significant bits),
plus the fp32 tolerance of the fp32 entry points, 1e-4 (1 + |y_ref|).

Covered: LayerNorm through the row kernel and the two-kernel path (vector and scalar
forms, long rows, misaligned pointers, in place, NULL affine, the full (16, 64, 256,
256) shape), RMSNorm (several channel counts, in place, the (2, 64, 32, 32)
workload), GroupNorm + LeakyReLU + x2 (vector and warp kernels, the (1024, 8192)
workload), GroupNorm over NCHW tensors (register kernel, clusters, two-kernel and
warp paths, the (8, 512, 64, 64) workload), and guard zones around every output.
"""
import numpy as np
import pytest
import torch

import normgen
import oracle
from gpu_util import assert_bf16_parity

pytestmark = pytest.mark.gpu

GUARD = 64
SENTINEL = 0x7FC1  # a bfloat16 NaN no kernel writes


@pytest.fixture(scope="module")
def ng():
    import memory_bound_normalization_norm_gb300 as m
    yield m
    m.norm_set_option(m.NORM_OPT_LN_PATH, 0)
    m.norm_set_option(m.NORM_OPT_GN_PATH, 0)
    m.norm_set_option(m.NORM_OPT_GN_CLUSTER, 0)


class BGuarded:
    """A bfloat16 device buffer of n elements between two guard zones of SENTINEL."""

    def __init__(self, n: int, init=None, offset: int = 0):
        self.n, self.lo = int(n), GUARD + offset
        bits = np.full(self.n + 2 * GUARD + offset, SENTINEL, dtype=np.uint16)
        if init is not None:
            bits[self.lo:self.lo + self.n] = normgen.bf16_bits(init)
        self.buf = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        self.t = self.buf[self.lo:self.lo + self.n]

    def values(self) -> np.ndarray:
        return normgen.bf16_to_f32(self.t.view(torch.int16).cpu().numpy().view(np.uint16))

    def guards_intact(self) -> bool:
        bits = self.buf.view(torch.int16).cpu().numpy().view(np.uint16)
        return bool((bits[:self.lo] == SENTINEL).all() and (bits[self.lo + self.n:] == SENTINEL).all())


def bf16_inputs(n, mean=0.0, std=1.0, seed=0, tensor_id=0):
    return normgen.round_bf16(normgen.normal(n, mean, std, seed=seed, tensor_id=tensor_id))


# ------------------------------------------------------------------ LayerNorm

def run_ln(ng, x, g, b, rows, L, path=0, offset=0, inplace=False):
    ng.norm_set_option(ng.NORM_OPT_LN_PATH, path)
    try:
        xb = BGuarded(rows * L, x, offset)
        gb = None if g is None else BGuarded(L, g, offset).t
        bb = None if b is None else BGuarded(L, b, offset).t
        yb = xb if inplace else BGuarded(rows * L, offset=offset)
        ng.norm_layer_fwd_bf16(xb.t, gb, bb, yb.t, rows, L, 1e-5)
        assert ng.norm_last_error() == 0
    finally:
        ng.norm_set_option(ng.NORM_OPT_LN_PATH, 0)
    assert yb.guards_intact(), "LayerNorm bf16 wrote outside its output"
    return yb.values()


@pytest.mark.parametrize("rows,L,path", [
    (3, 12, 3), (64, 4096, 3), (9, 16384, 3), (5, 1000, 3),   # row kernel
    (64, 4096, 4), (5, 20000, 4), (2, 131072, 4), (3, 65544, 4),  # streamed cluster kernel
    (2, 262144, 4), (3, 32768, 0),                                # bf16 slices of 4,096 packed vectors
    (2, 16388, 2), (3, 4096, 2), (2, 1 << 20, 2),             # two-kernel path, vector form
    (3, 1001, 0),                                             # two-kernel path, scalar form
])
def test_layer_norm_bf16(ng, rows, L, path):
    x = bf16_inputs(rows * L, seed=rows + L)
    g = bf16_inputs(L, 1.0, 0.1, seed=rows + L, tensor_id=1)
    b = bf16_inputs(L, 0.0, 0.1, seed=rows + L, tensor_id=2)
    want = oracle.layer_norm(x, g, b, rows, L, f64=True)
    assert_bf16_parity(run_ln(ng, x, g, b, rows, L, path=path), want, f"LN bf16 {rows}x{L} path={path}")


@pytest.mark.parametrize("offset", [0, 1])
def test_layer_norm_bf16_in_place_no_affine_misaligned(ng, offset):
    rows, L = 7, 2048
    x = bf16_inputs(rows * L, 2.0, 3.0, seed=11)
    want = oracle.layer_norm(x, None, None, rows, L, f64=True)
    assert_bf16_parity(run_ln(ng, x, None, None, rows, L, offset=offset), want, f"LN bf16 offset={offset}")
    assert_bf16_parity(run_ln(ng, x, None, None, rows, L, offset=offset, inplace=True), want,
                       f"LN bf16 in place offset={offset}")


@pytest.mark.parametrize("rows,L,path", [
    (2, 1 << 20, 0),       # the automatic choice above 131,072: one row group per row
    (3, 131080, 1),        # just above the cluster kernel's longest row (forced: the automatic choice
                           # takes the two-kernel path below 24 MiB)
    (16, 262144, 1),       # 16 row groups (a bf16 group row must stream as long as an fp32 one)
    (64, 262144, 0),       # 32 MiB of rows of 262,144: the automatic choice
    (2048, 32768, 0),      # 128 MiB of rows of 32,768: the automatic choice, 152 groups of 1 CTA
    (40, 131088, 1),       # forced: many row groups of few CTAs
    (5, 64, 1),            # forced: 8 units a row, most CTAs hold nothing
    (3, 8, 1),             # forced: one unit a row
    (1, (1 << 23) + 8, 0), # 8,388,616 values: 55,184 a CTA, close to the longest row
])
def test_layer_norm_bf16_persistent(ng, rows, L, path):
    """bf16 rows on the persistent kernel: 16-byte units of 8 values, gamma/beta packed in TMEM."""
    x = bf16_inputs(rows * L, seed=rows + L + 1)
    g = bf16_inputs(L, 1.0, 0.1, seed=rows + L + 1, tensor_id=1)
    b = bf16_inputs(L, 0.0, 0.1, seed=rows + L + 1, tensor_id=2)
    want = oracle.layer_norm(x, g, b, rows, L, f64=True)
    assert_bf16_parity(run_ln(ng, x, g, b, rows, L, path=path), want, f"LN bf16 persistent {rows}x{L} path={path}")


def test_layer_norm_bf16_persistent_no_affine_in_place_offset_mean(ng):
    rows, L = 3, 1 << 18
    x = bf16_inputs(rows * L, 50.0, 1.0, seed=12)  # bf16 spacing at 50 is 0.25: values well away from the mean's zero
    want = oracle.layer_norm(x, None, None, rows, L, f64=True)
    assert_bf16_parity(run_ln(ng, x, None, None, rows, L, path=1), want, "LN bf16 persistent no affine")
    assert_bf16_parity(run_ln(ng, x, None, None, rows, L, path=1, inplace=True), want,
                       "LN bf16 persistent in place")


@pytest.mark.parametrize("L,offset", [(131076, 0), (1 << 18, 4)])
def test_layer_norm_bf16_persistent_refusals(ng, L, offset):
    """Forced, the persistent kernel refuses rows that are not whole 16-byte units (L % 8 != 0) and
    tensors that are not 16-byte aligned (an offset of 4 elements); the automatic choice serves both."""
    rows = 2
    x = bf16_inputs(rows * L, seed=13)
    ng.norm_set_option(ng.NORM_OPT_LN_PATH, 1)
    try:
        xb, yb = BGuarded(rows * L, x, offset), BGuarded(rows * L, offset=offset)
        with pytest.raises(ng.NormError) as e:
            ng.norm_layer_fwd_bf16(xb.t, None, None, yb.t, rows, L, 1e-5)
        assert e.value.status == ng.NORM_ERR_UNSUPPORTED
    finally:
        ng.norm_set_option(ng.NORM_OPT_LN_PATH, 0)
    want = oracle.layer_norm(x, None, None, rows, L, f64=True)
    assert_bf16_parity(run_ln(ng, x, None, None, rows, L, offset=offset), want, f"LN bf16 {L} offset={offset}")


def test_layer_norm_bf16_full_size(ng):
    rows, L = 16, 64 * 256 * 256
    x = bf16_inputs(rows * L, seed=0)
    g = bf16_inputs(L, 1.0, 0.1, seed=0, tensor_id=1)
    b = bf16_inputs(L, 0.0, 0.1, seed=0, tensor_id=2)
    want = oracle.layer_norm(x, g, b, rows, L, f64=True)
    assert_bf16_parity(run_ln(ng, x, g, b, rows, L), want, "LN bf16 (16, 64, 256, 256)")


# ------------------------------------------------------------------ RMSNorm

@pytest.mark.parametrize("B,C,S", [(2, 64, 1024), (3, 1, 37), (2, 3, 129), (2, 128, 300), (2, 200, 65), (1, 48, 513),
                                   (2, 32, 1000), (3, 16, 2), (2, 64, 40002), (4, 8, 6), (2, 4, 258)])
def test_rms_bf16(ng, B, C, S):
    """Even S with C in {4, 8, 16, 32, 64} takes two positions a thread (4-byte loads and stores of
    bf16 pairs); odd S, other C and misaligned pointers take one position a thread."""
    x = bf16_inputs(B * C * S, seed=B * C + S)
    want = oracle.rms_channel(x, B, C, S, f64=True)
    xb, yb = BGuarded(B * C * S, x), BGuarded(B * C * S)
    ng.norm_rms_channel_fwd_bf16(xb.t, yb.t, B, C, S, 1e-5)
    assert ng.norm_last_error() == 0
    assert_bf16_parity(yb.values(), want, f"RMS bf16 ({B},{C},{S})")
    assert yb.guards_intact()
    ng.norm_rms_channel_fwd_bf16(xb.t, xb.t, B, C, S, 1e-5)
    assert_bf16_parity(xb.values(), want, f"RMS bf16 in place ({B},{C},{S})")


# ------------------------------------------------------------------ GroupNorm + LeakyReLU + x2

@pytest.mark.parametrize("N,C,G", [(7, 16 * 32, 32), (5, 4 * 8, 8), (3, 128 * 4, 4), (6, 3 * 16, 16),
                                   (4, 48 * 5, 5), (9, 64, 64), (1024, 8192, 512)])
def test_group_norm_bf16(ng, N, C, G):
    x = bf16_inputs(N * C, seed=N + C)
    g = bf16_inputs(C, 1.0, 0.1, seed=N + C, tensor_id=1)
    b = bf16_inputs(C, 0.0, 0.1, seed=N + C, tensor_id=2)
    want = oracle.group_lrelu_x2(x, g, b, N, C, G, f64=True)
    xb, gb, bb, yb = BGuarded(N * C, x), BGuarded(C, g), BGuarded(C, b), BGuarded(N * C)
    ng.norm_group_lrelu_x2_fwd_bf16(xb.t, gb.t, bb.t, yb.t, N, C, G, 1e-5, 0.01)
    assert ng.norm_last_error() == 0
    assert_bf16_parity(yb.values(), want, f"GN bf16 ({N},{C})/{G}")
    assert yb.guards_intact()


@pytest.mark.parametrize("M,G,N", [(8, 325, 13), (16, 163, 13), (32, 81, 13), (64, 41, 13), (128, 21, 13),
                                   (16, 64, 4099)])
@pytest.mark.parametrize("offset", [0, 4])
def test_group_norm_bf16_vector_forms(ng, M, G, N, offset):
    """Power-of-two groups of 8-128 channels: 16-byte aligned tensors take the 8-channel form
    (one 16-byte access a thread, four rows ahead), 8-byte aligned ones (offset 4) the
    4-channel form.  The widths leave a ragged last column block; (4099, 1024) walks about
    seven rows a CTA, past the rows in flight."""
    C = M * G
    x = bf16_inputs(N * C, seed=M + G + offset)
    g = bf16_inputs(C, 1.0, 0.1, seed=M + G + offset, tensor_id=1)
    b = bf16_inputs(C, 0.0, 0.1, seed=M + G + offset, tensor_id=2)
    want = oracle.group_lrelu_x2(x, g, b, N, C, G, f64=True)
    xb, gb, bb = BGuarded(N * C, x, offset), BGuarded(C, g, offset), BGuarded(C, b, offset)
    yb = BGuarded(N * C, offset=offset)
    ng.norm_group_lrelu_x2_fwd_bf16(xb.t, gb.t, bb.t, yb.t, N, C, G, 1e-5, 0.01)
    assert ng.norm_last_error() == 0
    assert_bf16_parity(yb.values(), want, f"GN bf16 ({N},{C})/{G} offset={offset}")
    assert yb.guards_intact()


@pytest.mark.parametrize("slope", [-0.5, 0.0, 1.0, 1.5])
def test_group_norm_bf16_vector_slopes_no_affine_in_place(ng, slope):
    N, C, G = 21, 16 * 96, 96
    x = bf16_inputs(N * C, 3.0, 2.0, seed=31)
    g = bf16_inputs(C, 1.0, 0.1, seed=31, tensor_id=1)
    b = bf16_inputs(C, 0.0, 0.1, seed=31, tensor_id=2)
    want = oracle.group_lrelu_x2(x, g, b, N, C, G, slope=slope, f64=True)
    xb, gb, bb, yb = BGuarded(N * C, x), BGuarded(C, g), BGuarded(C, b), BGuarded(N * C)
    ng.norm_group_lrelu_x2_fwd_bf16(xb.t, gb.t, bb.t, yb.t, N, C, G, 1e-5, slope)
    assert ng.norm_last_error() == 0
    assert_bf16_parity(yb.values(), want, f"GN bf16 slope={slope}")
    # no affine, in place
    want = oracle.group_lrelu_x2(x, None, None, N, C, G, slope=slope, f64=True)
    xb = BGuarded(N * C, x)
    ng.norm_group_lrelu_x2_fwd_bf16(xb.t, None, None, xb.t, N, C, G, 1e-5, slope)
    assert ng.norm_last_error() == 0
    assert_bf16_parity(xb.values(), want, f"GN bf16 no affine in place slope={slope}")
    assert xb.guards_intact()


def test_rms_bf16_misaligned(ng):
    # x and y 2-byte but not 4-byte aligned
    B, C, S = 2, 64, 1024
    x = bf16_inputs(B * C * S, seed=77)
    want = oracle.rms_channel(x, B, C, S, f64=True)
    xb, yb = BGuarded(B * C * S, x, offset=1), BGuarded(B * C * S, offset=1)
    ng.norm_rms_channel_fwd_bf16(xb.t, yb.t, B, C, S, 1e-5)
    assert ng.norm_last_error() == 0
    assert_bf16_parity(yb.values(), want, "RMS bf16 misaligned")
    assert yb.guards_intact()


def test_bf16_entry_points_check_dtype(ng):
    x = torch.zeros(64, device="cuda")
    with pytest.raises(TypeError):
        ng.norm_rms_channel_fwd_bf16(x, x, 1, 4, 16, 1e-5)


# ------------------------------------------------------------------ GroupNorm over NCHW

@pytest.mark.parametrize("N,C,S,G,path,cluster", [
    (2, 32, 64, 8, 1, 0),         # register kernel, one CTA per group
    (2, 32, 64, 8, 0, 0),         # team kernel (L = 256), the automatic choice
    (2, 8, 6, 4, 0, 0),           # team kernel, channels change inside a vector
    (2, 256, 4, 1, 5, 0),         # team kernel, 256 vectors a group
    (4, 240, 1, 6, 5, 0),         # team kernel, S = 1, M = 40
    (3, 30, 1, 1, 5, 0),          # team kernel, pairs of elements (M = 30)
    (3, 9, 5, 3, 5, 0),           # team kernel, single elements (L = 15)
    (2, 64, 1024, 4, 0, 0),       # automatic cluster of 2
    (1, 3, 2732, 1, 1, 16),       # forced cluster of 16, ragged slices
    (8, 512, 4096, 32, 0, 0),     # the (8, 512, 64, 64) 32-group workload: streamed, groups split over 8 CTAs
    (16, 512, 2048, 32, 0, 0),    # 512 groups of 32,768: split over 4 CTAs instead of the 2 that hold one
    (8, 512, 2048, 32, 0, 0),     # 256 groups of 32,768: the doubled split declined (one wave over clusters of 2)
    (16, 512, 4096, 32, 0, 0),    # 512 groups of 65,536: split over 8 CTAs
    (8, 512, 4096, 32, 1, 0),     # the same through the unstreamed register kernel
    (64, 64, 1024, 16, 4, 1),     # streamed, one CTA per group, many groups per CTA
    (2, 64, 1024, 4, 4, 16),      # streamed over clusters of 16
    (2, 16, 2046, 4, 4, 2),       # streamed, channels change inside a vector (L = 8184)
    (2, 64, 1024, 4, 4, 1),       # streamed, one CTA holding 4,096 packed vectors
    (3, 64, 300, 2, 4, 2),        # streamed, S = 300 < 4 * NT: a step is 3 channels and 124 values
    (2, 16, 1020, 1, 4, 0),       # streamed, S = 1020: a step is 1 channel and 4 values
    (100, 32, 4096, 4, 4, 2),     # streamed, full slices, S >= 4 * NT (the check-free copy), 1-2 groups a cluster
    (1, 32, 16384, 2, 0, 0),      # L = 262,144: 16 CTAs of 4,096 packed vectors
    (1, 128, 65536, 32, 0, 0),    # two-kernel path, vector form
    (3, 9, 5, 3, 2, 0),           # two-kernel path, scalar form
    (3, 9, 5, 3, 3, 0),           # warp path
])
def test_group_norm_nchw_bf16(ng, N, C, S, G, path, cluster):
    n = N * C * S
    x = bf16_inputs(n, seed=N + C + S)
    g = bf16_inputs(C, 1.0, 0.1, seed=N + C + S, tensor_id=1)
    b = bf16_inputs(C, 0.0, 0.1, seed=N + C + S, tensor_id=2)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, f64=True)
    xb, gb, bb, yb = BGuarded(n, x), BGuarded(C, g), BGuarded(C, b), BGuarded(n)
    ng.norm_set_option(ng.NORM_OPT_GN_PATH, path)
    ng.norm_set_option(ng.NORM_OPT_GN_CLUSTER, cluster)
    try:
        ng.norm_group_lrelu_x2_nchw_fwd_bf16(xb.t, gb.t, bb.t, yb.t, N, C, S, G, 1e-5, 0.01)
        assert ng.norm_last_error() == 0
    finally:
        ng.norm_set_option(ng.NORM_OPT_GN_PATH, 0)
        ng.norm_set_option(ng.NORM_OPT_GN_CLUSTER, 0)
    assert_bf16_parity(yb.values(), want, f"GN NCHW bf16 ({N},{C},{S})/{G}")
    assert yb.guards_intact()
    # in place
    ng.norm_group_lrelu_x2_nchw_fwd_bf16(xb.t, gb.t, bb.t, xb.t, N, C, S, G, 1e-5, 0.01)
    assert_bf16_parity(xb.values(), want, f"GN NCHW bf16 in place ({N},{C},{S})/{G}")


@pytest.mark.parametrize("N,C,S,G,path", [
    (1, 128, 512 * 512, 32, 0),  # (1, 128, 512, 512): 67 MB of x, the automatic choice
    (1, 128, 65536, 32, 6),      # forced: 32 segments of 262,144
    (2, 8, 36000, 2, 6),         # forced: S = 36000, a channel boundary inside a thread's stride
    (2, 2048, 8, 16, 6),         # forced: S = 8, a new channel at every unit
])
def test_group_norm_nchw_bf16_persistent(ng, N, C, S, G, path):
    n = N * C * S
    x = bf16_inputs(n, seed=N + C + S + 5)
    g = bf16_inputs(C, 1.0, 0.1, seed=N + C + S + 5, tensor_id=1)
    b = bf16_inputs(C, 0.0, 0.1, seed=N + C + S + 5, tensor_id=2)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, f64=True)
    xb, gb, bb, yb = BGuarded(n, x), BGuarded(C, g), BGuarded(C, b), BGuarded(n)
    ng.norm_set_option(ng.NORM_OPT_GN_PATH, path)
    try:
        ng.norm_group_lrelu_x2_nchw_fwd_bf16(xb.t, gb.t, bb.t, yb.t, N, C, S, G, 1e-5, 0.01)
        assert ng.norm_last_error() == 0
    finally:
        ng.norm_set_option(ng.NORM_OPT_GN_PATH, 0)
    assert_bf16_parity(yb.values(), want, f"GN NCHW bf16 persistent ({N},{C},{S})/{G}")
    assert yb.guards_intact()


def test_group_norm_nchw_bf16_persistent_refuses_split_units(ng):
    # S = 4: an 8-value unit would hold two channels
    N, C, S, G = 2, 64, 4, 4
    xb, yb = BGuarded(N * C * S, bf16_inputs(N * C * S, seed=3)), BGuarded(N * C * S)
    ng.norm_set_option(ng.NORM_OPT_GN_PATH, 6)
    try:
        with pytest.raises(ng.NormError) as e:
            ng.norm_group_lrelu_x2_nchw_fwd_bf16(xb.t, None, None, yb.t, N, C, S, G, 1e-5, 0.01)
        assert e.value.status == ng.NORM_ERR_UNSUPPORTED
    finally:
        ng.norm_set_option(ng.NORM_OPT_GN_PATH, 0)
