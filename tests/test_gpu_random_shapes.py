"""Seeded random shapes through every entry point's automatic path choice, against the
float64 oracle element by element, with guard zones around every output.

Shapes are drawn so that each operation's paths are all reached: LayerNorm rows from 1 to
300,000 elements (row kernel, cluster kernel, two-kernel path, persistent kernel at 2^20),
RMSNorm channel counts on both sides of the register kernels' limits, GroupNorm groups of
any size on (N, C) and NCHW tensors.  Each case also draws fp32 or bf16, a misaligned or
aligned placement (4-element misalignment turns the vector paths off) and in place or not.
The bf16 bound adds the rounding of the result (2^-8 |y|) to the fp32 one.
"""
import numpy as np
import pytest
import torch

import normgen
import oracle

pytestmark = pytest.mark.gpu

GUARD = 64
CASES = 80


@pytest.fixture(scope="module")
def ng():
    import memory_bound_normalization_norm_gb300 as m
    return m


class Buf:
    """n elements of fp32 or bf16 between guard zones of a NaN pattern no kernel writes."""

    def __init__(self, n, init, bf16, offset):
        self.n, self.bf16, self.lo = int(n), bf16, GUARD + offset
        total = self.n + 2 * GUARD + offset
        if bf16:
            bits = np.full(total, 0x7FC1, dtype=np.uint16)
            if init is not None:
                bits[self.lo:self.lo + self.n] = normgen.bf16_bits(init)
            self.buf = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        else:
            bits = np.full(total, 0x7FC0DEAD, dtype=np.uint32)
            if init is not None:
                bits[self.lo:self.lo + self.n] = np.asarray(init, dtype=np.float32).view(np.uint32)
            self.buf = torch.from_numpy(bits.view(np.int32)).cuda().view(torch.float32)
        self.t = self.buf[self.lo:self.lo + self.n]

    def values(self):
        if self.bf16:
            return normgen.bf16_to_f32(self.t.view(torch.int16).cpu().numpy().view(np.uint16))
        return self.t.cpu().numpy()

    def guards_intact(self):
        if self.bf16:
            bits = self.buf.view(torch.int16).cpu().numpy().view(np.uint16)
            s = 0x7FC1
        else:
            bits = self.buf.view(torch.int32).cpu().numpy().view(np.uint32)
            s = 0x7FC0DEAD
        return bool((bits[:self.lo] == s).all() and (bits[self.lo + self.n:] == s).all())


def check(got, want, bf16, what):
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    want = np.asarray(want, dtype=np.float64).reshape(-1)
    bound = 1e-4 * (1.0 + np.abs(want)) + (2.0**-8 * np.abs(want) if bf16 else 0.0)
    bad = ~(np.abs(got - want) <= bound)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {got.size} out of bound"


def draw_inputs(rng, n, c, seed, bf16):
    mean = float(rng.choice([0.0, 0.0, 3.0, -50.0]))
    std = float(rng.choice([1.0, 0.5, 4.0]))
    x = normgen.normal(n, mean, std, seed=seed, tensor_id=0)
    g = normgen.normal(c, 1.0, 0.1, seed=seed, tensor_id=1)
    b = normgen.normal(c, 0.0, 0.1, seed=seed, tensor_id=2)
    if bf16:
        x, g, b = normgen.round_bf16(x), normgen.round_bf16(g), normgen.round_bf16(b)
    if rng.random() < 0.2:
        g = b = None
    return x, g, b


def layouts(rng):
    bf16 = bool(rng.random() < 0.4)
    offset = int(rng.choice([0, 0, 0, 1]))
    inplace = bool(rng.random() < 0.3)
    return bf16, offset, inplace


@pytest.mark.parametrize("case", range(CASES))
def test_layer_norm_random(ng, case):
    rng = np.random.default_rng(1000 + case)
    L = int(rng.choice([int(rng.integers(1, 64)), int(rng.integers(64, 8193)), int(rng.integers(8193, 131073)),
                        int(rng.integers(131073, 300000)), 1 << 20]))
    rows = max(1, min(int(rng.integers(1, 40)), 4_000_000 // L))
    bf16, offset, inplace = layouts(rng)
    x, g, b = draw_inputs(rng, rows * L, L, 1000 + case, bf16)
    want = oracle.layer_norm(x, g, b, rows, L, f64=True)
    xb = Buf(rows * L, x, bf16, offset)
    gb = None if g is None else Buf(L, g, bf16, offset).t
    bb = None if b is None else Buf(L, b, bf16, offset).t
    yb = xb if inplace else Buf(rows * L, None, bf16, offset)
    fn = ng.norm_layer_fwd_bf16 if bf16 else ng.norm_layer_fwd
    fn(xb.t, gb, bb, yb.t, rows, L, 1e-5)
    assert ng.norm_last_error() == 0
    check(yb.values(), want, bf16, f"LN case {case}: {rows}x{L} bf16={bf16} offset={offset} inplace={inplace}")
    assert yb.guards_intact()


@pytest.mark.parametrize("case", range(CASES))
def test_rms_random(ng, case):
    rng = np.random.default_rng(2000 + case)
    C = int(rng.choice([int(rng.integers(1, 17)), int(rng.integers(17, 65)), int(rng.integers(65, 129)),
                        int(rng.integers(129, 300))]))
    S = int(rng.integers(1, 5000))
    B = max(1, min(int(rng.integers(1, 6)), 2_000_000 // (C * S)))
    bf16, offset, inplace = layouts(rng)
    x, _, _ = draw_inputs(rng, B * C * S, 1, 2000 + case, bf16)
    want = oracle.rms_channel(x, B, C, S, f64=True)
    xb = Buf(B * C * S, x, bf16, offset)
    yb = xb if inplace else Buf(B * C * S, None, bf16, offset)
    fn = ng.norm_rms_channel_fwd_bf16 if bf16 else ng.norm_rms_channel_fwd
    fn(xb.t, yb.t, B, C, S, 1e-5)
    assert ng.norm_last_error() == 0
    check(yb.values(), want, bf16, f"RMS case {case}: ({B},{C},{S}) bf16={bf16} offset={offset} inplace={inplace}")
    assert yb.guards_intact()


@pytest.mark.parametrize("case", range(CASES))
def test_group_norm_random(ng, case):
    rng = np.random.default_rng(3000 + case)
    M = int(rng.choice([1, 2, 3, 4, 8, 16, 32, 48, 64, 128, 256, 1000, int(rng.integers(1, 5000))]))
    G = int(rng.integers(1, 40))
    nchw = bool(rng.random() < 0.6)
    S = int(rng.choice([1, 4, 7, 64, 1024, 4096, int(rng.integers(1, 3000))])) if nchw else 1
    while M * S > 300_000:
        S = max(1, S // 4)
    C = M * G
    N = max(1, min(int(rng.integers(1, 12)), 3_000_000 // (C * S)))
    slope = float(rng.choice([0.01, 0.2, 0.0]))
    bf16, offset, inplace = layouts(rng)
    x, g, b = draw_inputs(rng, N * C * S, C, 3000 + case, bf16)
    want = oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G, 1e-5, slope, f64=True)
    xb = Buf(N * C * S, x, bf16, offset)
    gb = None if g is None else Buf(C, g, bf16, offset).t
    bb = None if b is None else Buf(C, b, bf16, offset).t
    yb = xb if inplace else Buf(N * C * S, None, bf16, offset)
    if nchw:
        fn = ng.norm_group_lrelu_x2_nchw_fwd_bf16 if bf16 else ng.norm_group_lrelu_x2_nchw_fwd
        fn(xb.t, gb, bb, yb.t, N, C, S, G, 1e-5, slope)
    else:
        fn = ng.norm_group_lrelu_x2_fwd_bf16 if bf16 else ng.norm_group_lrelu_x2_fwd
        fn(xb.t, gb, bb, yb.t, N, C, G, 1e-5, slope)
    assert ng.norm_last_error() == 0
    check(yb.values(), want, bf16,
          f"GN case {case}: N={N} C={C} S={S} G={G} nchw={nchw} bf16={bf16} offset={offset} inplace={inplace}")
    assert yb.guards_intact()
