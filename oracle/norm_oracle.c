/*
 * norm_oracle.c - TEST INFRASTRUCTURE: the plain, slow CPU float64 oracle.
 *
 * Only the test suite, __graft_entry__.smoke() and the CPU-baseline /
 * reference arm of bench.py may load or run this code.  The CUDA library
 * shares no code, header, table or helper with it, and neither includes
 * the other.
 *
 * Every function takes the fp32 input bytes the GPU sees (for the Linear:
 * the bfloat16 values of x and W, widened exactly to float), promotes them to
 * double, evaluates the operation's textbook definition in double with an
 * explicit two-pass variance, and writes the result in double (y64) and/or
 * rounded once to float (y32).  Either output pointer may be NULL.
 * `threads` only splits independent units (rows, batch entries, samples)
 * across OpenMP threads; the arithmetic inside a unit is sequential and in
 * the order written here.
 *
 * Sources (the three web pages the method is taken from):
 *  - LayerNorm: POPCORNBENCH transcript "Kimi-K2.6 l1_p40", opening problem
 *    analysis: per batch element, mean and population variance (unbiased =
 *    False) over the last three dims; y = (x - mean) / sqrt(var + eps) *
 *    weight + bias with elementwise weight/bias of the normalized shape.
 *  - GroupNorm + LeakyReLU + x+x: transcript "Kimi-K2.6 l2_p62", first
 *    design turn: groups of C/G contiguous channels, var = sum((x-mean)^2)/M,
 *    y = (x - mean)/sqrt(var + eps) * gamma_c + beta_c, LeakyReLU(t) =
 *    max(0, t) + negative_slope * min(0, t), then x + x.
 *    The same operation over x[N][C][S] (an NCHW tensor with S = H*W): a
 *    group holds its M channels at every spatial position, M*S values,
 *    which are contiguous in memory; gamma/beta stay per channel.
 *  - RMSNorm: transcript "Kimi-K2.6 l1_p36", reference model quoted in the
 *    analysis turn: rms = sqrt(mean(x^2, dim=1) + eps), y = x / rms, over
 *    dim 1 of an NCHW tensor whose trailing dims flatten to S = H*W.
 *  - Linear, then GroupNorm + LeakyReLU + x+x: transcript "Kimi-K2.6
 *    l2_p62", the module and its forward as the page writes them:
 *    h = F.linear(x, W, b) = x W^T + b with W [out][in] as nn.Linear stores
 *    it, then the GroupNorm + LeakyReLU + x+x above on each row of h (the
 *    page's first design turn weighs computing the group statistics in the
 *    GEMM's epilogue).
 *
 * Pins (tests/test_oracle_pins.py): exact rational brute force on tiny
 * inputs, closed forms (constant rows, affine invariance, two-valued rows,
 * one-hot and constant RMS positions, GroupNorm with one channel per group
 * as worked on the GroupNorm page), invariants of the outputs, float64
 * torch.nn.functional on CPU as a third voice, and planted-mistake
 * (mutation) runs that every pin set must catch.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG -1

static void oracle_store(double v, int64_t i, double *y64, float *y32)
{
    if (y64)
        y64[i] = v;
    if (y32)
        y32[i] = (float)v;
}

/* LayerNorm over contiguous rows x[rows][L]; gamma/beta [L] or NULL
 * (identity affine: weight 1, bias 0). */
int oracle_layer_norm(const float *x, const float *gamma, const float *beta,
                      int64_t rows, int64_t L, double eps,
                      double *y64, float *y32, int threads)
{
    if (!x || rows < 0 || L <= 0 || !(eps >= 0.0) || (!y64 && !y32))
        return ORACLE_BAD_ARG;
    if (threads < 1)
        threads = 1;
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * L;
        /* pass 1: mean */
        double sum = 0.0;
        for (int64_t i = 0; i < L; ++i)
            sum += (double)xr[i];
        const double mean = sum / (double)L;
        /* pass 2: population variance about the mean */
        double sq = 0.0;
        for (int64_t i = 0; i < L; ++i) {
            const double d = (double)xr[i] - mean;
            sq += d * d;
        }
        const double var = sq / (double)L;
        const double denom = sqrt(var + eps);
        for (int64_t i = 0; i < L; ++i) {
            const double w = gamma ? (double)gamma[i] : 1.0;
            const double b = beta ? (double)beta[i] : 0.0;
            const double v = ((double)xr[i] - mean) / denom * w + b;
            oracle_store(v, r * L + i, y64, y32);
        }
    }
    return ORACLE_OK;
}

/* RMSNorm over dim 1 of x[B][C][S] (S = product of the trailing dims), no
 * affine: for each (b, s), ms = (1/C) sum_c x[b][c][s]^2,
 * rms = sqrt(ms + eps), y[b][c][s] = x[b][c][s] / rms. */
int oracle_rms_channel(const float *x, int64_t B, int64_t C, int64_t S, double eps,
                       double *y64, float *y32, int threads)
{
    if (!x || B < 0 || C <= 0 || S < 0 || !(eps >= 0.0) || (!y64 && !y32))
        return ORACLE_BAD_ARG;
    if (threads < 1)
        threads = 1;
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1)
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t s = 0; s < S; ++s) {
            const float *xp = x + b * C * S + s;
            double sq = 0.0;
            for (int64_t c = 0; c < C; ++c) {
                const double v = (double)xp[c * S];
                sq += v * v;
            }
            const double rms = sqrt(sq / (double)C + eps);
            for (int64_t c = 0; c < C; ++c)
                oracle_store((double)xp[c * S] / rms, b * C * S + c * S + s, y64, y32);
        }
    }
    return ORACLE_OK;
}

/* GroupNorm over x[N][C] with G groups of M = C/G contiguous channels
 * (group g holds channels g*M .. g*M+M-1), per-channel gamma/beta [C] or
 * NULL (weight 1, bias 0), population variance, then
 * LeakyReLU(t) = max(0, t) + slope * min(0, t), then out = l + l. */
int oracle_group_lrelu_x2(const float *x, const float *gamma, const float *beta,
                          int64_t N, int64_t C, int64_t G, double eps, double slope,
                          double *y64, float *y32, int threads)
{
    if (!x || N < 0 || C <= 0 || G <= 0 || C % G != 0 || !(eps >= 0.0) || (!y64 && !y32))
        return ORACLE_BAD_ARG;
    if (threads < 1)
        threads = 1;
    const int64_t M = C / G;
#pragma omp parallel for num_threads(threads) schedule(dynamic, 16)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < G; ++g) {
            const int64_t c0 = g * M;
            const float *xg = x + n * C + c0;
            double sum = 0.0;
            for (int64_t j = 0; j < M; ++j)
                sum += (double)xg[j];
            const double mean = sum / (double)M;
            double sq = 0.0;
            for (int64_t j = 0; j < M; ++j) {
                const double d = (double)xg[j] - mean;
                sq += d * d;
            }
            const double var = sq / (double)M;
            const double denom = sqrt(var + eps);
            for (int64_t j = 0; j < M; ++j) {
                const int64_t c = c0 + j;
                const double w = gamma ? (double)gamma[c] : 1.0;
                const double b = beta ? (double)beta[c] : 0.0;
                const double t = ((double)xg[j] - mean) / denom * w + b;
                const double l = fmax(0.0, t) + slope * fmin(0.0, t);
                oracle_store(l + l, n * C + c, y64, y32);
            }
        }
    }
    return ORACLE_OK;
}

/* GroupNorm + LeakyReLU + x+x over x[N][C][S]: group g of sample n holds
 * channels g*M .. g*M+M-1 (M = C/G) at all S positions, i.e. the M*S values
 * x[n][c][s]; mean and population variance over them; then per element
 * t = (x - mean) / sqrt(var + eps) * gamma[c] + beta[c] (gamma/beta [C] or
 * NULL), LeakyReLU, out = l + l.  S = 1 is oracle_group_lrelu_x2. */
int oracle_group_lrelu_x2_nchw(const float *x, const float *gamma, const float *beta,
                               int64_t N, int64_t C, int64_t S, int64_t G, double eps, double slope,
                               double *y64, float *y32, int threads)
{
    if (!x || N < 0 || C <= 0 || S <= 0 || G <= 0 || C % G != 0 || !(eps >= 0.0) || (!y64 && !y32))
        return ORACLE_BAD_ARG;
    if (threads < 1)
        threads = 1;
    const int64_t M = C / G;
    const double cnt = (double)(M * S);
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < G; ++g) {
            const int64_t c0 = g * M;
            double sum = 0.0;
            for (int64_t c = c0; c < c0 + M; ++c)
                for (int64_t s = 0; s < S; ++s)
                    sum += (double)x[(n * C + c) * S + s];
            const double mean = sum / cnt;
            double sq = 0.0;
            for (int64_t c = c0; c < c0 + M; ++c)
                for (int64_t s = 0; s < S; ++s) {
                    const double d = (double)x[(n * C + c) * S + s] - mean;
                    sq += d * d;
                }
            const double denom = sqrt(sq / cnt + eps);
            for (int64_t c = c0; c < c0 + M; ++c) {
                const double gw = gamma ? (double)gamma[c] : 1.0;
                const double bw = beta ? (double)beta[c] : 0.0;
                for (int64_t s = 0; s < S; ++s) {
                    const int64_t i = (n * C + c) * S + s;
                    const double v = ((double)x[i] - mean) / denom * gw + bw;
                    const double l = fmax(0.0, v) + slope * fmin(0.0, v);
                    oracle_store(l + l, i, y64, y32);
                }
            }
        }
    }
    return ORACLE_OK;
}

/* Linear, then GroupNorm + LeakyReLU + x+x.  x[Mr][K] (rows), w[N][K] (the
 * Linear's weight, one row per output channel), bias [N] or NULL (0):
 *     h[m][n] = sum_k x[m][k] * w[n][k] + bias[n]
 * in double, summed in order of k; then each row h[m][0..N-1] goes through
 * the GroupNorm + LeakyReLU + x+x of oracle_group_lrelu_x2 (G groups of N/G
 * contiguous channels, gamma/beta [N] or NULL), with h kept in double. */
int oracle_linear_group_lrelu_x2(const float *x, const float *w, const float *bias,
                                 const float *gamma, const float *beta,
                                 int64_t Mr, int64_t K, int64_t N, int64_t G, double eps, double slope,
                                 double *y64, float *y32, int threads)
{
    if (!x || !w || Mr < 0 || K <= 0 || N <= 0 || G <= 0 || N % G != 0 || !(eps >= 0.0) ||
        (!y64 && !y32))
        return ORACLE_BAD_ARG;
    if (threads < 1)
        threads = 1;
    const int64_t M = N / G;
    int bad = 0;
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1)
    for (int64_t m = 0; m < Mr; ++m) {
        double *h = (double *)malloc((size_t)N * sizeof(double));
        if (!h) {
#pragma omp atomic write
            bad = 1;
            continue;
        }
        const float *xm = x + m * K;
        /* the Linear: one dot product of length K per output channel */
        for (int64_t n = 0; n < N; ++n) {
            const float *wn = w + n * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)xm[k] * (double)wn[k];
            h[n] = acc + (bias ? (double)bias[n] : 0.0);
        }
        /* GroupNorm over groups of M contiguous channels, then LeakyReLU, then x+x */
        for (int64_t g = 0; g < G; ++g) {
            const int64_t c0 = g * M;
            double sum = 0.0;
            for (int64_t j = 0; j < M; ++j)
                sum += h[c0 + j];
            const double mean = sum / (double)M;
            double sq = 0.0;
            for (int64_t j = 0; j < M; ++j) {
                const double d = h[c0 + j] - mean;
                sq += d * d;
            }
            const double denom = sqrt(sq / (double)M + eps);
            for (int64_t j = 0; j < M; ++j) {
                const int64_t c = c0 + j;
                const double gw = gamma ? (double)gamma[c] : 1.0;
                const double bw = beta ? (double)beta[c] : 0.0;
                const double t = (h[c] - mean) / denom * gw + bw;
                const double l = fmax(0.0, t) + slope * fmin(0.0, t);
                oracle_store(l + l, m * N + c, y64, y32);
            }
        }
        free(h);
    }
    return bad ? ORACLE_BAD_ARG : ORACLE_OK;
}
