"""The Linear + GroupNorm + LeakyReLU + x2 kernel (tensor-core GEMM with the
normalization in its epilogue) against the float64 oracle, element by element.

Inputs are bfloat16 x and W (the values the tensor cores read; the oracle gets
the same values widened exactly) and fp32 bias/gamma/beta, drawn as the
GroupNorm page's module draws them: nn.Linear's default init, W and bias ~
U(-1/sqrt(K), 1/sqrt(K)), and gamma ~ N(1, 0.1), beta ~ N(0, 0.1).  The bound is
the fp32 one, |y - y_ref| <= 1e-4 (1 + |y_ref|): products of bfloat16 values
are exact in fp32 and only the fp32 accumulation order differs.

Covered: one tile and many; several tiles per CTA (both TMEM accumulators in
turn); rows and channels past a 128 x 256 tile edge; K not a multiple of the
64-wide stage; groups of 16, 32 and 64; NULL bias/gamma/beta; several slopes;
two calls in a row; the page's full (1024, 8192) x Linear(8192, 8192), 512
groups; and the shapes the kernel refuses.
"""
import numpy as np
import pytest
import torch

import normgen
import oracle
from gpu_util import TOL, assert_parity, bf16_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ng():
    import memory_bound_normalization_norm_gb300 as m
    return m


def inputs(M, K, N, seed):
    bound = K ** -0.5
    x = normgen.round_bf16(normgen.normal(M * K, seed=seed, tensor_id=normgen.TENSOR_X))
    w = normgen.round_bf16(normgen.uniform(N * K, -bound, bound, seed=seed, tensor_id=normgen.TENSOR_W))
    bias = normgen.uniform(N, -bound, bound, seed=seed, tensor_id=normgen.TENSOR_LIN_BIAS)
    g = normgen.normal(N, 1.0, 0.1, seed=seed, tensor_id=normgen.TENSOR_GAMMA)
    b = normgen.normal(N, 0.0, 0.1, seed=seed, tensor_id=normgen.TENSOR_BETA)
    return x, w, bias, g, b


def run(ng, x, w, bias, g, b, M, K, N, G, slope=0.01):
    dev = torch.device("cuda")
    f32 = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    y = torch.full((M * N + 64,), float("nan"), dtype=torch.float32, device=dev)
    ng.norm_linear_group_lrelu_x2_fwd(bf16_device(x), bf16_device(w), f32(bias), f32(g), f32(b), y, M, K, N, G,
                                      1e-5, slope)
    assert ng.norm_last_error() == ng.NORM_OK
    out = y.cpu().numpy()
    assert np.isnan(out[M * N:]).all(), "wrote past the end of y"
    return out[:M * N]


def check(ng, M, K, N, G, seed, slope=0.01, affine=True):
    x, w, bias, g, b = inputs(M, K, N, seed)
    if not affine:
        bias = g = b = None
    want = oracle.linear_group_lrelu_x2(x, w, bias, g, b, M, K, N, G, 1e-5, slope)
    got = run(ng, x, w, bias, g, b, M, K, N, G, slope)
    return assert_parity(got, want, f"Linear+GN M={M} K={K} N={N} G={G} slope={slope}", TOL)


@pytest.mark.parametrize("M,K,N,G", [
    (128, 64, 256, 16),     # one tile, one stage
    (128, 256, 256, 16),    # one tile, the ring of stages wraps
    (256, 512, 1024, 64),   # 8 tiles
    (200, 192, 256, 16),    # rows past the tile edge
    (130, 72, 272, 17),     # K not a multiple of 64; channels past the tile edge
    (64, 128, 512, 16),     # fewer rows than one tile
    (256, 128, 512, 16),    # groups of 32 (G = 16)
    (384, 136, 768, 12),    # groups of 64
])
def test_shapes(ng, M, K, N, G):
    check(ng, M, K, N, G, seed=M + K + N + G)


def test_several_tiles_per_cta(ng):
    # 16 x 32 = 512 tiles over at most one CTA per SM: both accumulators in turn
    check(ng, 2048, 64, 8192, 512, seed=3)


@pytest.mark.parametrize("slope", [0.0, 0.2, 1.0, -0.5])
def test_slopes(ng, slope):
    check(ng, 256, 128, 512, 32, seed=4, slope=slope)


def test_no_affine_no_bias(ng):
    check(ng, 256, 128, 512, 32, seed=5, affine=False)


def test_two_calls_in_a_row(ng):
    M, K, N, G = 512, 256, 1024, 64
    x, w, bias, g, b = inputs(M, K, N, 6)
    want = oracle.linear_group_lrelu_x2(x, w, bias, g, b, M, K, N, G, 1e-5, 0.01)
    for k in range(2):
        assert_parity(run(ng, x, w, bias, g, b, M, K, N, G), want, f"call {k + 1}", TOL)


@pytest.mark.slow
def test_full_size(ng):
    """The GroupNorm page's module: x (1024, 8192), Linear(8192, 8192), 512 groups of 16."""
    check(ng, 1024, 8192, 8192, 512, seed=0)


def test_refusals(ng):
    dev = torch.device("cuda")
    x = torch.zeros(256 * 64, dtype=torch.bfloat16, device=dev)
    w = torch.zeros(256 * 64, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(256 * 256, dtype=torch.float32, device=dev)
    raw = ng.raw()
    call = lambda M, K, N, G, xp=x.data_ptr(), yp=y.data_ptr(): raw.norm_linear_group_lrelu_x2_fwd(  # noqa: E731
        xp, w.data_ptr(), None, None, None, yp, M, K, N, G, 1e-5, 0.01, torch.cuda.current_stream().cuda_stream)
    assert call(128, 64, 256, 32) == ng.NORM_ERR_UNSUPPORTED      # groups of 8
    assert call(128, 60, 256, 16) == ng.NORM_ERR_UNSUPPORTED      # K not a multiple of 8
    assert call(128, 64, 256, 3) == ng.NORM_ERR_INVALID_ARG       # 256 % 3 != 0
    assert call(128, 64, 256, 16, xp=x.data_ptr() + 2) == ng.NORM_ERR_UNSUPPORTED  # x not 16-byte aligned
    assert call(0, 64, 256, 16) == ng.NORM_OK                     # empty
    torch.cuda.synchronize()
    assert float(y.abs().max()) == 0.0
