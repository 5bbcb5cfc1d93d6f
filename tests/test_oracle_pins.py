"""The oracle against its pins, and planted mistakes that the pins must catch.

A planted mistake is a one-place textual change to a copy of ``oracle/norm_oracle.c``
(a dropped term, a wrong sign, index or divisor, a transposed operand), compiled
on the CPU into a temporary library.  Each one must make at least one pin of its
operation fail; a mistake no pin catches would mean the oracle is not pinned.
"""
import numpy as np
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("op", sorted(ALL_PINS))
def test_oracle_meets_its_pins(op):
    ALL_PINS[op](oracle.get())


# (operation, name, text in norm_oracle.c, replacement).  Every replacement keeps all
# memory accesses in bounds.
MUTANTS = [
    ("layer_norm", "unbiased variance", "const double var = sq / (double)L;", "const double var = sq / (double)(L + 1);"),
    ("layer_norm", "mean off by one", "const double mean = sum / (double)L;\n        /* pass 2",
     "const double mean = sum / (double)(L + 1);\n        /* pass 2"),
    ("layer_norm", "eps outside sqrt", "const double denom = sqrt(var + eps);\n        for (int64_t i = 0; i < L; ++i) {",
     "const double denom = sqrt(var) + eps;\n        for (int64_t i = 0; i < L; ++i) {"),
    ("layer_norm", "eps dropped", "const double denom = sqrt(var + eps);\n        for (int64_t i = 0; i < L; ++i) {",
     "const double denom = sqrt(var + 1e-12);\n        for (int64_t i = 0; i < L; ++i) {"),
    ("layer_norm", "bias dropped", "const double v = ((double)xr[i] - mean) / denom * w + b;",
     "const double v = ((double)xr[i] - mean) / denom * w;"),
    ("layer_norm", "sign flipped", "const double v = ((double)xr[i] - mean) / denom * w + b;",
     "const double v = (mean - (double)xr[i]) / denom * w + b;"),
    ("layer_norm", "weight reversed", "const double w = gamma ? (double)gamma[i] : 1.0;\n            const double b = beta ? (double)beta[i] : 0.0;\n            const double v",
     "const double w = gamma ? (double)gamma[L - 1 - i] : 1.0;\n            const double b = beta ? (double)beta[i] : 0.0;\n            const double v"),
    ("layer_norm", "weight and bias swapped", "const double w = gamma ? (double)gamma[i] : 1.0;\n            const double b = beta ? (double)beta[i] : 0.0;\n            const double v",
     "const double w = beta ? (double)beta[i] : 1.0;\n            const double b = gamma ? (double)gamma[i] : 0.0;\n            const double v"),
    ("layer_norm", "variance not centred", "const double d = (double)xr[i] - mean;\n            sq += d * d;\n        }\n        const double var = sq / (double)L;",
     "const double d = (double)xr[i];\n            sq += d * d;\n        }\n        const double var = sq / (double)L;"),
    ("layer_norm", "stats from row 0", "const float *xr = x + r * L;\n        /* pass 1",
     "const float *xr = x + 0 * L;\n        /* pass 1"),
    ("rms_channel", "eps dropped", "const double rms = sqrt(sq / (double)C + eps);", "const double rms = sqrt(sq / (double)C);"),
    ("rms_channel", "sum instead of mean", "const double rms = sqrt(sq / (double)C + eps);", "const double rms = sqrt(sq + eps);"),
    ("rms_channel", "multiply by rms", "oracle_store((double)xp[c * S] / rms,", "oracle_store((double)xp[c * S] * rms,"),
    ("rms_channel", "output transposed", "oracle_store((double)xp[c * S] / rms, b * C * S + c * S + s, y64, y32);",
     "oracle_store((double)xp[c * S] / rms, b * C * S + s * C + c, y64, y32);"),
    ("rms_channel", "reduce over positions", "const double v = (double)xp[c * S];",
     "const double v = (double)x[b * C * S + (s + c) % S];"),
    ("rms_channel", "mean not squared", "sq += v * v;\n            }\n            const double rms",
     "sq += v;\n            }\n            const double rms"),
    ("group_lrelu_x2", "strided groups", "for (int64_t j = 0; j < M; ++j)\n                sum += (double)xg[j];",
     "for (int64_t j = 0; j < M; ++j)\n                sum += (double)x[n * C + g + j * G];"),
    ("group_lrelu_x2", "unbiased variance", "const double var = sq / (double)M;", "const double var = sq / (double)(M + 1);"),
    ("group_lrelu_x2", "eps outside sqrt", "const double denom = sqrt(var + eps);\n            for (int64_t j",
     "const double denom = sqrt(var) + eps;\n            for (int64_t j"),
    ("group_lrelu_x2", "slope on positive side",
     "const double l = fmax(0.0, t) + slope * fmin(0.0, t);\n                oracle_store(l + l, n * C + c",
     "const double l = slope * fmax(0.0, t) + fmin(0.0, t);\n                oracle_store(l + l, n * C + c"),
    ("group_lrelu_x2", "x+x dropped", "oracle_store(l + l, n * C + c, y64, y32);", "oracle_store(l, n * C + c, y64, y32);"),
    ("group_lrelu_x2", "gamma per group", "const double w = gamma ? (double)gamma[c] : 1.0;", "const double w = gamma ? (double)gamma[g] : 1.0;"),
    ("group_lrelu_x2", "beta dropped", "const double t = ((double)xg[j] - mean) / denom * w + b;",
     "const double t = ((double)xg[j] - mean) / denom * w;"),
    ("group_lrelu_x2", "relu before affine", "const double t = ((double)xg[j] - mean) / denom * w + b;\n                const double l = fmax(0.0, t) + slope * fmin(0.0, t);",
     "const double u = ((double)xg[j] - mean) / denom;\n                const double t = (fmax(0.0, u) + slope * fmin(0.0, u)) * w + b;\n                const double l = t;"),
    ("group_lrelu_x2_nchw", "count M, not M*S", "const double cnt = (double)(M * S);", "const double cnt = (double)M;"),
    ("group_lrelu_x2_nchw", "positions read as channels", "sum += (double)x[(n * C + c) * S + s];",
     "sum += (double)x[(n * S + s) * C + c];"),
    ("group_lrelu_x2_nchw", "eps outside sqrt", "const double denom = sqrt(sq / cnt + eps);",
     "const double denom = sqrt(sq / cnt) + eps;"),
    ("group_lrelu_x2_nchw", "gamma per group",
     "const double gw = gamma ? (double)gamma[c] : 1.0;\n                const double bw = beta ? (double)beta[c] : 0.0;\n                for (int64_t s",
     "const double gw = gamma ? (double)gamma[c0] : 1.0;\n                const double bw = beta ? (double)beta[c] : 0.0;\n                for (int64_t s"),
    ("group_lrelu_x2_nchw", "beta per position", "const double v = ((double)x[i] - mean) / denom * gw + bw;",
     "const double v = ((double)x[i] - mean) / denom * gw + (beta ? (double)beta[(c0 + s) % C] : 0.0);"),
    ("group_lrelu_x2_nchw", "slope on positive side", "fmax(0.0, v) + slope * fmin(0.0, v)",
     "slope * fmax(0.0, v) + fmin(0.0, v)"),
    ("group_lrelu_x2_nchw", "x+x dropped", "oracle_store(l + l, i, y64, y32);", "oracle_store(l, i, y64, y32);"),
    ("linear_group_lrelu_x2", "weight transposed", "acc += (double)xm[k] * (double)wn[k];",
     "acc += (double)xm[k] * (double)w[(k * N + n) % (N * K)];"),
    ("linear_group_lrelu_x2", "last k skipped", "for (int64_t k = 0; k < K; ++k)\n                acc +=",
     "for (int64_t k = 0; k < K - 1; ++k)\n                acc +="),
    ("linear_group_lrelu_x2", "bias dropped", "h[n] = acc + (bias ? (double)bias[n] : 0.0);", "h[n] = acc;"),
    ("linear_group_lrelu_x2", "bias by row", "h[n] = acc + (bias ? (double)bias[n] : 0.0);",
     "h[n] = acc + (bias ? (double)bias[m % N] : 0.0);"),
    ("linear_group_lrelu_x2", "x row 0 for every row", "const float *xm = x + m * K;", "const float *xm = x + 0 * K;"),
    ("linear_group_lrelu_x2", "strided groups", "sum += h[c0 + j];", "sum += h[(g + j * G) % N];"),
    ("linear_group_lrelu_x2", "unbiased variance", "sqrt(sq / (double)M + eps)", "sqrt(sq / (double)(M + 1) + eps)"),
    ("linear_group_lrelu_x2", "gamma per group", "const double gw = gamma ? (double)gamma[c] : 1.0;\n                const double bw = beta ? (double)beta[c] : 0.0;\n                const double t = (h[c]",
     "const double gw = gamma ? (double)gamma[g] : 1.0;\n                const double bw = beta ? (double)beta[c] : 0.0;\n                const double t = (h[c]"),
    ("linear_group_lrelu_x2", "slope on positive side",
     "const double l = fmax(0.0, t) + slope * fmin(0.0, t);\n                oracle_store(l + l, m * N + c",
     "const double l = slope * fmax(0.0, t) + fmin(0.0, t);\n                oracle_store(l + l, m * N + c"),
    ("linear_group_lrelu_x2", "x+x dropped", "oracle_store(l + l, m * N + c, y64, y32);", "oracle_store(l, m * N + c, y64, y32);"),
    ("group_lrelu_x2_nchw", "variance about zero", "const double d = (double)x[(n * C + c) * S + s] - mean;",
     "const double d = (double)x[(n * C + c) * S + s];"),
]


@pytest.mark.parametrize("op,name,find,repl", MUTANTS, ids=[f"{m[0]}:{m[1]}" for m in MUTANTS])
def test_planted_mistake_is_caught(op, name, find, repl, tmp_path):
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(find) == 1, f"mutation anchor for '{name}' must occur exactly once"
    bad = oracle.build_variant(src.replace(find, repl), str(tmp_path))
    with pytest.raises(AssertionError):
        with np.errstate(all="ignore"):
            ALL_PINS[op](bad)
