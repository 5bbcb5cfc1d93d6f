"""Pins for the float64 oracle: checks that tie it to something other than itself.

Each ``*_pins(o)`` runs every check for one operation against an ``oracle.Oracle``
handle and raises ``AssertionError`` naming the first check that fails.  The same
functions run against the committed oracle (all must pass) and against builds with
a planted mistake (at least one must fail), see ``test_oracle_pins.py``.

Kinds of pin:
  * exact brute force: tiny inputs of small dyadic rationals, statistics in exact
    ``fractions.Fraction`` arithmetic and the square root in 60-digit ``decimal``;
  * closed forms: constant rows/groups, affine invariance, two-valued rows,
    one-hot and constant RMS positions, one channel per group (the worked case on
    the GroupNorm page, stored under ``golden/``);
  * invariants of the outputs (zero mean, known variance, known mean square);
  * float64 ``torch.nn.functional`` on CPU as a third voice on small shapes.
"""
from __future__ import annotations

import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np

import normgen

getcontext().prec = 60
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

EPS = 1e-5


# ----------------------------------------------------------------------------- exact helpers

def _dec(fr: Fraction) -> Decimal:
    return Decimal(fr.numerator) / Decimal(fr.denominator)


def _dsqrt(fr: Fraction) -> Decimal:
    return _dec(fr).sqrt()


def _dyadic(rng, shape, k=64, den=16):
    """Small dyadic rationals j/den, |j| <= k: exact in fp32 and in double."""
    return (rng.integers(-k, k + 1, size=shape) / den).astype(np.float32)


def _close(got, want, tol, what):
    got = np.asarray(got, dtype=np.float64).ravel()
    want = np.asarray(want, dtype=np.float64).ravel()
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    if not np.all(np.isfinite(got)):
        raise AssertionError(f"{what}: non-finite output")
    err = np.abs(got - want) / (1.0 + np.abs(want))
    i = int(np.argmax(err))
    assert err[i] <= tol, f"{what}: scaled error {err[i]:.3e} > {tol:.1e} at {i} (got {got[i]!r}, want {want[i]!r})"


def exact_layer_norm(x, gamma, beta, rows, L, eps):
    x = np.asarray(x, dtype=np.float32).reshape(rows, L)
    out = np.empty((rows, L), dtype=np.float64)
    fe = Fraction(eps)
    for r in range(rows):
        xs = [Fraction(float(v)) for v in x[r]]
        mean = sum(xs) / L
        var = sum((v - mean) ** 2 for v in xs) / L
        den = _dsqrt(var + fe)
        for i, v in enumerate(xs):
            w = Fraction(float(gamma[i])) if gamma is not None else Fraction(1)
            b = Fraction(float(beta[i])) if beta is not None else Fraction(0)
            out[r, i] = float(_dec(v - mean) / den * _dec(w) + _dec(b))
    return out


def exact_rms_channel(x, B, C, S, eps):
    x = np.asarray(x, dtype=np.float32).reshape(B, C, S)
    out = np.empty((B, C, S), dtype=np.float64)
    fe = Fraction(eps)
    for b in range(B):
        for s in range(S):
            xs = [Fraction(float(x[b, c, s])) for c in range(C)]
            ms = sum(v * v for v in xs) / C
            rms = _dsqrt(ms + fe)
            for c in range(C):
                out[b, c, s] = float(_dec(xs[c]) / rms)
    return out


def exact_group_lrelu_x2(x, gamma, beta, N, C, G, eps, slope):
    x = np.asarray(x, dtype=np.float32).reshape(N, C)
    M = C // G
    out = np.empty((N, C), dtype=np.float64)
    fe, fs = Fraction(eps), Fraction(slope)
    for n in range(N):
        for g in range(G):
            xs = [Fraction(float(v)) for v in x[n, g * M:(g + 1) * M]]
            mean = sum(xs) / M
            var = sum((v - mean) ** 2 for v in xs) / M
            den = _dsqrt(var + fe)
            for j, v in enumerate(xs):
                c = g * M + j
                w = Fraction(float(gamma[c])) if gamma is not None else Fraction(1)
                b = Fraction(float(beta[c])) if beta is not None else Fraction(0)
                t = _dec(v - mean) / den * _dec(w) + _dec(b)
                l = t if t > 0 else _dec(fs) * t
                out[n, c] = float(l + l)
    return out


def exact_group_lrelu_x2_nchw(x, gamma, beta, N, C, S, G, eps, slope):
    x = np.asarray(x, dtype=np.float32).reshape(N, C, S)
    M = C // G
    out = np.empty((N, C, S), dtype=np.float64)
    fe, fs = Fraction(eps), Fraction(slope)
    for n in range(N):
        for g in range(G):
            xs = [[Fraction(float(v)) for v in x[n, c]] for c in range(g * M, (g + 1) * M)]
            flat = [v for row in xs for v in row]
            mean = sum(flat) / (M * S)
            var = sum((v - mean) ** 2 for v in flat) / (M * S)
            den = _dsqrt(var + fe)
            for j in range(M):
                c = g * M + j
                w = Fraction(float(gamma[c])) if gamma is not None else Fraction(1)
                b = Fraction(float(beta[c])) if beta is not None else Fraction(0)
                for s_ in range(S):
                    t = _dec(xs[j][s_] - mean) / den * _dec(w) + _dec(b)
                    l = t if t > 0 else _dec(fs) * t
                    out[n, c, s_] = float(l + l)
    return out


def exact_linear_group_lrelu_x2(x, w, bias, gamma, beta, Mr, K, N, G, eps, slope):
    """h = x W^T + bias exactly (Fractions), then the GroupNorm + LeakyReLU + x+x of each row of h."""
    x = np.asarray(x, dtype=np.float32).reshape(Mr, K)
    w = np.asarray(w, dtype=np.float32).reshape(N, K)
    M = N // G
    out = np.empty((Mr, N), dtype=np.float64)
    fe, fs = Fraction(eps), Fraction(slope)
    for m in range(Mr):
        h = []
        for n in range(N):
            acc = sum(Fraction(float(x[m, k])) * Fraction(float(w[n, k])) for k in range(K))
            h.append(acc + (Fraction(float(bias[n])) if bias is not None else Fraction(0)))
        for g in range(G):
            hs = h[g * M:(g + 1) * M]
            mean = sum(hs) / M
            var = sum((v - mean) ** 2 for v in hs) / M
            den = _dsqrt(var + fe)
            for j, v in enumerate(hs):
                c = g * M + j
                gw = Fraction(float(gamma[c])) if gamma is not None else Fraction(1)
                bw = Fraction(float(beta[c])) if beta is not None else Fraction(0)
                t = _dec(v - mean) / den * _dec(gw) + _dec(bw)
                l = t if t > 0 else _dec(fs) * t
                out[m, c] = float(l + l)
    return out


# ----------------------------------------------------------------------------- LayerNorm

def layer_norm_pins(o) -> None:
    rng = np.random.default_rng(20240601)

    # 1. exact brute force, several rows (row indexing), affine and identity affine
    for L in (1, 2, 3, 5, 8):
        rows = 3
        x = _dyadic(rng, rows * L)
        g = _dyadic(rng, L, k=32, den=8)
        b = _dyadic(rng, L, k=32, den=8)
        for gg, bb in ((g, b), (None, None)):
            want = exact_layer_norm(x, gg, bb, rows, L, EPS)
            got = o.layer_norm(x, gg, bb, rows, L, EPS, f64=True)
            _close(got, want, 1e-11, f"LN brute force L={L} affine={gg is not None}")
            got32 = o.layer_norm(x, gg, bb, rows, L, EPS)
            assert np.array_equal(got32, got.astype(np.float32)), "LN fp32 output is not the double result rounded once"

    # 2. constant row -> y = beta exactly (variance 0, finite 1/sqrt(eps))
    L = 37
    g = _dyadic(rng, L, k=32, den=8)
    b = _dyadic(rng, L, k=32, den=8)
    for c in (0.0, -3.25, 1000.0):
        x = np.full(2 * L, c, dtype=np.float32)
        got = o.layer_norm(x, g, b, 2, L, EPS, f64=True)
        assert np.array_equal(got.reshape(2, L), np.stack([b, b]).astype(np.float64)), f"LN constant row {c}"

    # 3. affine invariance: LN(a*x + c) == LN(x) for a > 0 with eps = 0 (exact inputs),
    #    and within 1e-5 for eps = 1e-5 when a^2 var >> eps
    L = 1024
    x = _dyadic(rng, 2 * L, k=256, den=64)
    base = o.layer_norm(x, None, None, 2, L, 0.0, f64=True)
    for a in (0.5, 4.0, 1024.0):
        for c in (-7.0, 1024.0):
            xs = (np.float32(a) * x + np.float32(c)).astype(np.float32)
            assert np.array_equal(xs.astype(np.float64), a * x.astype(np.float64) + c), "inexact scaled input"
            _close(o.layer_norm(xs, None, None, 2, L, 0.0, f64=True), base, 1e-12, f"LN invariance a={a} c={c}")
    big = (np.float32(1024.0) * x).astype(np.float32)
    _close(o.layer_norm(big, None, None, 2, L, EPS, f64=True), base, 2e-5, "LN invariance with eps")

    # 4. two-valued row +a/-a in equal counts -> mean 0, var a^2, y = +-a/sqrt(a^2+eps)*g+b
    L = 64
    a = 0.375
    sign = np.where(np.arange(L) % 2 == 0, 1.0, -1.0)
    x = (a * sign).astype(np.float32)
    g = _dyadic(rng, L, k=32, den=8)
    b = _dyadic(rng, L, k=32, den=8)
    want = sign * a / np.sqrt(a * a + EPS) * g.astype(np.float64) + b.astype(np.float64)
    _close(o.layer_norm(x, g, b, 1, L, EPS, f64=True), want, 1e-14, "LN two-valued row")

    # 5. invariants on a random row: mean(y) = 0, population var(y) = var/(var+eps),
    #    and (y * sqrt(var+eps) + mean) reconstructs x
    L = 4099
    x = normgen.normal(3 * L, 3.0, 2.0, seed=1)
    y = o.layer_norm(x, None, None, 3, L, EPS, f64=True).reshape(3, L)
    xr = x.reshape(3, L).astype(np.float64)
    for r in range(3):
        mu = np.mean(xr[r])
        var = np.mean((xr[r] - mu) ** 2)
        assert abs(np.mean(y[r])) < 1e-12, "LN output mean not 0"
        assert abs(np.mean(y[r] ** 2) - var / (var + EPS)) < 1e-12, "LN output variance"
        _close(y[r] * np.sqrt(var + EPS) + mu, xr[r], 1e-13, "LN reconstruction")

    # 6. third voice: float64 torch.nn.functional.layer_norm over the last 3 dims
    import torch
    shape = (3, 5, 7, 11)
    L = 5 * 7 * 11
    x = normgen.normal(3 * L, 0.5, 1.5, seed=2)
    g = normgen.normal(L, 1.0, 0.1, seed=2, tensor_id=1)
    b = normgen.normal(L, 0.0, 0.1, seed=2, tensor_id=2)
    ref = torch.nn.functional.layer_norm(
        torch.from_numpy(x.astype(np.float64)).reshape(shape), shape[1:],
        torch.from_numpy(g.astype(np.float64)).reshape(shape[1:]),
        torch.from_numpy(b.astype(np.float64)).reshape(shape[1:]), EPS).numpy()
    _close(o.layer_norm(x, g, b, 3, L, EPS, f64=True), ref, 1e-12, "LN vs torch float64")


# ----------------------------------------------------------------------------- RMSNorm

def rms_channel_pins(o) -> None:
    rng = np.random.default_rng(20240602)

    # 1. exact brute force with B, C, S > 1 (catches transposed channel/position indexing)
    for (B, C, S) in ((1, 1, 1), (2, 3, 5), (2, 4, 3), (1, 8, 2)):
        x = _dyadic(rng, B * C * S)
        want = exact_rms_channel(x, B, C, S, EPS)
        got = o.rms_channel(x, B, C, S, EPS, f64=True)
        _close(got, want, 1e-12, f"RMS brute force {(B, C, S)}")
        assert np.array_equal(o.rms_channel(x, B, C, S, EPS), got.astype(np.float32)), "RMS fp32 rounding"

    # 2. one-hot position: value a in channel k -> y_k = a / sqrt(a^2/C + eps), others 0
    B, C, S = 2, 64, 9
    x = np.zeros((B, C, S), dtype=np.float32)
    a = np.float32(-2.5)
    x[1, 17, 4] = a
    y = o.rms_channel(x, B, C, S, EPS, f64=True).reshape(B, C, S)
    want = np.zeros_like(y)
    want[1, 17, 4] = float(a) / np.sqrt(float(a) ** 2 / C + EPS)
    _close(y, want, 1e-14, "RMS one-hot")

    # 3. constant position a -> y = a / sqrt(a^2 + eps); C = 1 -> x / sqrt(x^2 + eps)
    x = np.full((2, 6, 5), 0.75, dtype=np.float32)
    _close(o.rms_channel(x, 2, 6, 5, EPS, f64=True), np.full(60, 0.75 / np.sqrt(0.5625 + EPS)), 1e-14,
           "RMS constant position")
    x = _dyadic(rng, 40)
    xd = x.astype(np.float64)
    _close(o.rms_channel(x, 4, 1, 10, EPS, f64=True), xd / np.sqrt(xd * xd + EPS), 1e-14, "RMS C=1")

    # 4. invariant: mean_c(y^2) = ms / (ms + eps) at every position
    B, C, S = 3, 64, 257
    x = normgen.normal(B * C * S, seed=3)
    y = o.rms_channel(x, B, C, S, EPS, f64=True).reshape(B, C, S)
    xd = x.reshape(B, C, S).astype(np.float64)
    ms = np.mean(xd * xd, axis=1)
    assert np.max(np.abs(np.mean(y * y, axis=1) - ms / (ms + EPS))) < 1e-13, "RMS output mean square"

    # 5. third voice: torch.nn.functional.rms_norm over the channel dim of NHWC in float64
    import torch
    B, C, H, W = 2, 7, 3, 5
    x = normgen.normal(B * C * H * W, seed=4)
    t = torch.from_numpy(x.astype(np.float64)).reshape(B, C, H, W)
    ref = torch.nn.functional.rms_norm(t.permute(0, 2, 3, 1), (C,), eps=EPS).permute(0, 3, 1, 2)
    _close(o.rms_channel(x, B, C, H * W, EPS, f64=True), ref.contiguous().numpy(), 1e-13, "RMS vs torch")


# ----------------------------------------------------------------------------- GroupNorm + LeakyReLU + x+x

def read_golden_gn():
    rows = []
    with open(os.path.join(GOLDEN, "gn_one_channel_per_group.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(v) for v in line.split()])
    return np.array(rows, dtype=np.float64)


def group_lrelu_x2_pins(o) -> None:
    rng = np.random.default_rng(20240603)

    # 1. exact brute force: groups of contiguous channels, per-channel affine, two slopes
    for (N, C, G) in ((2, 8, 1), (2, 8, 2), (3, 8, 4), (1, 6, 3), (2, 12, 3)):
        x = _dyadic(rng, N * C)
        g = _dyadic(rng, C, k=32, den=8)
        b = _dyadic(rng, C, k=32, den=8)
        for slope in (0.01, 0.25):
            want = exact_group_lrelu_x2(x, g, b, N, C, G, EPS, slope)
            got = o.group_lrelu_x2(x, g, b, N, C, G, EPS, slope, f64=True)
            _close(got, want, 1e-11, f"GN brute force {(N, C, G)} slope={slope}")
        assert np.array_equal(o.group_lrelu_x2(x, g, b, N, C, G, EPS, 0.01),
                              o.group_lrelu_x2(x, g, b, N, C, G, EPS, 0.01, f64=True).astype(np.float32))

    # 2. one channel per group: the worked case on the GroupNorm page (golden file)
    gold = read_golden_gn()
    for row in gold:
        xv, gv, bv, slope, want = row
        got = o.group_lrelu_x2(np.array([xv], np.float32), np.array([gv], np.float32),
                               np.array([bv], np.float32), 1, 1, 1, EPS, slope, f64=True)
        assert got[0] == want, f"GN M=1 golden: got {got[0]!r}, want {want!r}"
    C = 16
    x = _dyadic(rng, 3 * C)
    g = _dyadic(rng, C, k=32, den=8)
    b = _dyadic(rng, C, k=32, den=8)
    bd = b.astype(np.float64)
    want = np.tile(2.0 * np.where(bd > 0, bd, 0.01 * bd), 3)
    _close(o.group_lrelu_x2(x, g, b, 3, C, C, EPS, 0.01, f64=True), want, 0.0, "GN M=1 -> 2*LReLU(beta)")

    # 3. constant group -> 2 * LReLU(beta)
    x = np.full(2 * 32, -1.5, dtype=np.float32)
    g = _dyadic(rng, 32, k=32, den=8)
    b = _dyadic(rng, 32, k=32, den=8)
    bd = b.astype(np.float64)
    _close(o.group_lrelu_x2(x, g, b, 2, 32, 4, EPS, 0.01, f64=True),
           np.tile(2.0 * np.where(bd > 0, bd, 0.01 * bd), 2), 0.0, "GN constant group")

    # 4. third voice: torch float64 group_norm -> leaky_relu -> x + x; slope 1 gives 2*GN
    import torch
    N, C, G = 4, 48, 6
    x = normgen.normal(N * C, seed=5)
    g = normgen.normal(C, 1.0, 0.1, seed=5, tensor_id=1)
    b = normgen.normal(C, 0.0, 0.1, seed=5, tensor_id=2)
    t = torch.nn.functional.group_norm(torch.from_numpy(x.astype(np.float64)).reshape(N, C), G,
                                       torch.from_numpy(g.astype(np.float64)),
                                       torch.from_numpy(b.astype(np.float64)), EPS)
    for slope in (0.01, 1.0):
        l = torch.nn.functional.leaky_relu(t, slope)
        _close(o.group_lrelu_x2(x, g, b, N, C, G, EPS, slope, f64=True), (l + l).numpy(), 1e-12,
               f"GN vs torch slope={slope}")

    # 5. invariant: with gamma=1, beta=0, slope=1 every group of y/2 has mean 0 and
    #    population variance var/(var+eps)
    N, C, G = 3, 64, 4
    x = normgen.normal(N * C, 2.0, 3.0, seed=6)
    y = o.group_lrelu_x2(x, None, None, N, C, G, EPS, 1.0, f64=True).reshape(N, G, C // G) / 2.0
    xd = x.astype(np.float64).reshape(N, G, C // G)
    var = np.mean((xd - xd.mean(axis=2, keepdims=True)) ** 2, axis=2)
    assert np.max(np.abs(y.mean(axis=2))) < 1e-13, "GN group mean"
    assert np.max(np.abs(np.mean(y * y, axis=2) - var / (var + EPS))) < 1e-12, "GN group variance"


# ----------------------------------------------------------------------------- GroupNorm over NCHW

def group_lrelu_x2_nchw_pins(o) -> None:
    rng = np.random.default_rng(20240917)

    # 1. exact brute force: a group is its M channels at every spatial position
    for (N, C, S, G) in ((2, 4, 3, 2), (1, 6, 2, 3), (2, 8, 1, 4), (1, 4, 5, 1), (2, 6, 4, 6)):
        x = _dyadic(rng, N * C * S)
        g = _dyadic(rng, C, k=32, den=8)
        b = _dyadic(rng, C, k=32, den=8)
        for slope in (0.01, 0.25):
            want = exact_group_lrelu_x2_nchw(x, g, b, N, C, S, G, EPS, slope).reshape(-1)
            got = o.group_lrelu_x2_nchw(x, g, b, N, C, S, G, EPS, slope, f64=True)
            _close(got, want, 1e-11, f"GN NCHW brute force {(N, C, S, G)} slope={slope}")

    # 2. S = 1 is the (N, C) operation, bit for bit
    N, C, G = 3, 48, 6
    x = normgen.normal(N * C, seed=8)
    g = normgen.normal(C, 1.0, 0.1, seed=8, tensor_id=1)
    b = normgen.normal(C, 0.0, 0.1, seed=8, tensor_id=2)
    assert np.array_equal(o.group_lrelu_x2_nchw(x, g, b, N, C, 1, G, EPS, 0.01, f64=True),
                          o.group_lrelu_x2(x, g, b, N, C, G, EPS, 0.01, f64=True)), "GN NCHW with S = 1"

    # 3. third voice: torch float64 group_norm on (N, C, H, W) -> leaky_relu -> x + x
    import torch
    N, C, H, W, G = 2, 12, 3, 5, 4
    x = normgen.normal(N * C * H * W, 0.5, 2.0, seed=9)
    g = normgen.normal(C, 1.0, 0.1, seed=9, tensor_id=1)
    b = normgen.normal(C, 0.0, 0.1, seed=9, tensor_id=2)
    t = torch.nn.functional.group_norm(torch.from_numpy(x.astype(np.float64)).reshape(N, C, H, W), G,
                                       torch.from_numpy(g.astype(np.float64)),
                                       torch.from_numpy(b.astype(np.float64)), EPS)
    for slope in (0.01, 1.0):
        l = torch.nn.functional.leaky_relu(t, slope)
        _close(o.group_lrelu_x2_nchw(x, g, b, N, C, H * W, G, EPS, slope, f64=True), (l + l).numpy().reshape(-1),
               1e-12, f"GN NCHW vs torch slope={slope}")

    # 4. invariant: gamma=1, beta=0, slope=1: y/2 over each group's M*S values has
    #    mean 0 and population variance var/(var+eps)
    N, C, S, G = 2, 16, 7, 4
    x = normgen.normal(N * C * S, -1.0, 3.0, seed=10)
    y = o.group_lrelu_x2_nchw(x, None, None, N, C, S, G, EPS, 1.0, f64=True).reshape(N, G, -1) / 2.0
    xd = x.astype(np.float64).reshape(N, G, -1)
    var = np.mean((xd - xd.mean(axis=2, keepdims=True)) ** 2, axis=2)
    assert np.max(np.abs(y.mean(axis=2))) < 1e-13, "GN NCHW group mean"
    assert np.max(np.abs(np.mean(y * y, axis=2) - var / (var + EPS))) < 1e-12, "GN NCHW group variance"

    # 5. constant group -> 2 * LReLU(beta) at every position of every channel
    x = np.full(2 * 8 * 5, 3.25, dtype=np.float32)
    g = _dyadic(rng, 8, k=32, den=8)
    b = _dyadic(rng, 8, k=32, den=8)
    bd = b.astype(np.float64)
    want = np.tile(np.repeat(2.0 * np.where(bd > 0, bd, 0.01 * bd), 5), 2)
    _close(o.group_lrelu_x2_nchw(x, g, b, 2, 8, 5, 2, EPS, 0.01, f64=True), want, 0.0, "GN NCHW constant group")


# ----------------------------------------------------------------------------- Linear + GroupNorm

def linear_group_lrelu_x2_pins(o) -> None:
    rng = np.random.default_rng(20241203)

    # 1. exact brute force: h = x W^T + bias in Fractions, then the group statistics
    for (Mr, K, N, G) in ((2, 3, 4, 2), (3, 5, 8, 4), (1, 8, 6, 3), (2, 4, 4, 1), (3, 2, 6, 6)):
        x = _dyadic(rng, Mr * K)
        w = _dyadic(rng, N * K, k=32, den=8)
        bias = _dyadic(rng, N, k=32, den=8)
        g = _dyadic(rng, N, k=32, den=8)
        b = _dyadic(rng, N, k=32, den=8)
        for slope in (0.01, 0.25):
            want = exact_linear_group_lrelu_x2(x, w, bias, g, b, Mr, K, N, G, EPS, slope).reshape(-1)
            got = o.linear_group_lrelu_x2(x, w, bias, g, b, Mr, K, N, G, EPS, slope, f64=True)
            _close(got, want, 1e-11, f"Linear+GN brute force {(Mr, K, N, G)} slope={slope}")
        assert np.array_equal(o.linear_group_lrelu_x2(x, w, bias, g, b, Mr, K, N, G, EPS, 0.01),
                              o.linear_group_lrelu_x2(x, w, bias, g, b, Mr, K, N, G, EPS, 0.01,
                                                      f64=True).astype(np.float32)), "Linear+GN fp32 rounding"

    # 2. reductions to the (pinned) GroupNorm oracle, bit for bit:
    #    a permutation weight (not symmetric) selects channels: h[m][n] = x[m][perm[n]]
    Mr, K, G = 5, 48, 6
    x = normgen.normal(Mr * K, seed=11)
    g = normgen.normal(K, 1.0, 0.1, seed=11, tensor_id=1)
    b = normgen.normal(K, 0.0, 0.1, seed=11, tensor_id=2)
    perm = rng.permutation(K)
    assert np.any(perm[perm] != np.arange(K)), "the permutation must not be its own inverse"
    w = np.zeros((K, K), dtype=np.float32)
    w[np.arange(K), perm] = 1.0
    want = o.group_lrelu_x2(x.reshape(Mr, K)[:, perm].copy(), g, b, Mr, K, G, EPS, 0.01, f64=True).reshape(-1)
    assert np.array_equal(o.linear_group_lrelu_x2(x, w, None, g, b, Mr, K, K, G, EPS, 0.01, f64=True), want), \
        "Linear+GN with a permutation weight"
    #    a zero weight leaves the bias: every row is the GroupNorm of the bias
    N = 24
    bias = normgen.normal(N, 0.0, 2.0, seed=12, tensor_id=4)
    g2 = normgen.normal(N, 1.0, 0.1, seed=12, tensor_id=1)
    b2 = normgen.normal(N, 0.0, 0.1, seed=12, tensor_id=2)
    want = o.group_lrelu_x2(np.tile(bias, 3), g2, b2, 3, N, 4, EPS, 0.01, f64=True)
    got = o.linear_group_lrelu_x2(normgen.normal(3 * 7, seed=13), np.zeros((N, 7), np.float32), bias, g2, b2,
                                  3, 7, N, 4, EPS, 0.01, f64=True)
    assert np.array_equal(got, want), "Linear+GN with a zero weight"

    # 3. third voice: float64 torch F.linear -> group_norm -> leaky_relu -> x + x
    import torch
    Mr, K, N, G = 6, 40, 32, 4
    x = normgen.normal(Mr * K, seed=14)
    w = normgen.uniform(N * K, -K ** -0.5, K ** -0.5, seed=14, tensor_id=3)
    bias = normgen.uniform(N, -K ** -0.5, K ** -0.5, seed=14, tensor_id=4)
    g = normgen.normal(N, 1.0, 0.1, seed=14, tensor_id=1)
    b = normgen.normal(N, 0.0, 0.1, seed=14, tensor_id=2)
    d = lambda a: torch.from_numpy(a.astype(np.float64))  # noqa: E731
    h = torch.nn.functional.linear(d(x).reshape(Mr, K), d(w).reshape(N, K), d(bias))
    t = torch.nn.functional.group_norm(h, G, d(g), d(b), EPS)
    for slope in (0.01, 1.0):
        l = torch.nn.functional.leaky_relu(t, slope)
        _close(o.linear_group_lrelu_x2(x, w, bias, g, b, Mr, K, N, G, EPS, slope, f64=True),
               (l + l).numpy().reshape(-1), 1e-12, f"Linear+GN vs torch slope={slope}")

    # 4. invariant: gamma=1, beta=0, slope=1: y/2 per group has mean 0 and population
    #    variance var/(var+eps), var taken from h = x W^T + bias (float64 matmul)
    Mr, K, N, G = 4, 24, 32, 8
    x = normgen.normal(Mr * K, 1.0, 2.0, seed=15)
    w = normgen.normal(N * K, seed=15, tensor_id=3)
    bias = normgen.normal(N, seed=15, tensor_id=4)
    y = o.linear_group_lrelu_x2(x, w, bias, None, None, Mr, K, N, G, EPS, 1.0, f64=True).reshape(Mr, G, -1) / 2.0
    hd = (x.astype(np.float64).reshape(Mr, K) @ w.astype(np.float64).reshape(N, K).T + bias).reshape(Mr, G, -1)
    var = np.mean((hd - hd.mean(axis=2, keepdims=True)) ** 2, axis=2)
    assert np.max(np.abs(y.mean(axis=2))) < 1e-13, "Linear+GN group mean"
    assert np.max(np.abs(np.mean(y * y, axis=2) - var / (var + EPS))) < 1e-12, "Linear+GN group variance"


ALL_PINS = {
    "layer_norm": layer_norm_pins,
    "rms_channel": rms_channel_pins,
    "group_lrelu_x2": group_lrelu_x2_pins,
    "group_lrelu_x2_nchw": group_lrelu_x2_nchw_pins,
    "linear_group_lrelu_x2": linear_group_lrelu_x2_pins,
}
