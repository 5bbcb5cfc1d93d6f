/*
 * normgen.c - seeded, counter-based synthetic input generator.
 *
 * This file is shared by the test oracle and the CUDA path's tests and
 * benchmark: both sides draw their inputs from here, so they see the same
 * fp32 bytes.  It holds none of the normalization arithmetic.
 *
 * Stream definition (SplitMix64, Steele/Lea/Flood 2014, as published by
 * S. Vigna): a SplitMix64 generator seeded with s0 returns as its k-th
 * output (k = 0, 1, ...)
 *
 *     word(k) = mix(s0 + (k + 1) * 0x9E3779B97F4A7C15)
 *     mix(z)  : z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *               z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
 *
 * Because word(k) depends only on (s0, k), any element of any tensor can be
 * produced on its own: the output is independent of the thread count and of
 * which sub-range is asked for.
 *
 * Per (seed, tensor_id) the stream seed is
 *     s0 = mix(mix(seed) ^ (tensor_id * 0xD1B54A32D192ED03 + 1)).
 *
 * Uniform draw from word w: u = ((w >> 11) + 0.5) * 2^-53, in (0, 1).
 * Normal draw (Box-Muller, 1958), element pairs (2p, 2p+1) share
 *     u1 = u(word(2p)), u2 = u(word(2p+1)),
 *     r = sqrt(-2 ln u1), th = 2 pi u2,
 *     z(2p) = r cos th, z(2p+1) = r sin th,
 * and element i of a N(mean, std^2) tensor is (float)(mean + std * z(i)),
 * computed in double and rounded once.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#define NG_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t ng_mix(uint64_t z)
{
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

static inline uint64_t ng_word(uint64_t s0, uint64_t k)
{
    return ng_mix(s0 + (k + 1ULL) * NG_GAMMA);
}

static inline double ng_unit(uint64_t w)
{
    return ((double)(w >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

uint64_t normgen_stream_seed(uint64_t seed, uint64_t tensor_id)
{
    return ng_mix(ng_mix(seed) ^ (tensor_id * 0xD1B54A32D192ED03ULL + 1ULL));
}

/* k-th output of a SplitMix64 generator seeded with s0 (for known-answer tests). */
uint64_t normgen_splitmix64_output(uint64_t s0, uint64_t k)
{
    return ng_word(s0, k);
}

uint64_t normgen_word(uint64_t seed, uint64_t tensor_id, uint64_t k)
{
    return ng_word(normgen_stream_seed(seed, tensor_id), k);
}

/* z(i) of the standard normal stream. */
static inline double ng_normal(uint64_t s0, uint64_t i)
{
    const uint64_t p = i >> 1;
    const double u1 = ng_unit(ng_word(s0, 2 * p));
    const double u2 = ng_unit(ng_word(s0, 2 * p + 1));
    const double r = sqrt(-2.0 * log(u1));
    const double th = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? r * sin(th) : r * cos(th);
}

enum { NG_NORMAL = 0, NG_UNIFORM = 1 };

typedef struct {
    int kind;
    uint64_t s0;
    uint64_t start;
    int64_t begin, end; /* this worker's slice of [0, n) */
    double a, b;        /* normal: mean, std.  uniform: lo, hi */
    float *out;
} ng_job;

static void ng_run(const ng_job *j)
{
    if (j->kind == NG_NORMAL) {
        int64_t i = j->begin;
        /* Pairs share their two uniforms; compute both members at once. */
        while (i < j->end) {
            const uint64_t gi = j->start + (uint64_t)i;
            if ((gi & 1) == 0 && i + 1 < j->end) {
                const uint64_t p = gi >> 1;
                const double u1 = ng_unit(ng_word(j->s0, 2 * p));
                const double u2 = ng_unit(ng_word(j->s0, 2 * p + 1));
                const double r = sqrt(-2.0 * log(u1));
                const double th = 6.283185307179586476925286766559 * u2;
                j->out[i] = (float)(j->a + j->b * (r * cos(th)));
                j->out[i + 1] = (float)(j->a + j->b * (r * sin(th)));
                i += 2;
            } else {
                j->out[i] = (float)(j->a + j->b * ng_normal(j->s0, gi));
                i += 1;
            }
        }
    } else {
        for (int64_t i = j->begin; i < j->end; ++i) {
            const double u = ng_unit(ng_word(j->s0, j->start + (uint64_t)i));
            j->out[i] = (float)(j->a + (j->b - j->a) * u);
        }
    }
}

static void *ng_thread(void *arg)
{
    ng_run((const ng_job *)arg);
    return NULL;
}

static int ng_fill(int kind, uint64_t seed, uint64_t tensor_id, uint64_t start,
                   int64_t n, double a, double b, float *out, int threads)
{
    if (n < 0 || (n > 0 && out == NULL))
        return -1;
    if (threads < 1)
        threads = 1;
    if (threads > 256)
        threads = 256;
    if (n < 65536)
        threads = 1;
    const uint64_t s0 = normgen_stream_seed(seed, tensor_id);
    ng_job jobs[256];
    pthread_t tids[256];
    int started[256];
    for (int t = 0; t < threads; ++t) {
        /* Split on even boundaries so Box-Muller pairs stay together. */
        int64_t lo = (int64_t)(((__int128)n * t) / threads) & ~(int64_t)1;
        int64_t hi = (t == threads - 1) ? n : ((int64_t)(((__int128)n * (t + 1)) / threads) & ~(int64_t)1);
        if (t == 0)
            lo = 0;
        jobs[t].kind = kind;
        jobs[t].s0 = s0;
        jobs[t].start = start;
        jobs[t].begin = lo;
        jobs[t].end = hi;
        jobs[t].a = a;
        jobs[t].b = b;
        jobs[t].out = out;
        started[t] = 0;
    }
    for (int t = 1; t < threads; ++t)
        started[t] = pthread_create(&tids[t], NULL, ng_thread, &jobs[t]) == 0;
    ng_run(&jobs[0]);
    for (int t = 1; t < threads; ++t) {
        if (started[t])
            pthread_join(tids[t], NULL);
        else
            ng_run(&jobs[t]);
    }
    return 0;
}

/* out[i] = (float)(mean + std * z(start + i)), i in [0, n). Returns 0 on success. */
int normgen_fill_normal(uint64_t seed, uint64_t tensor_id, uint64_t start, int64_t n,
                        double mean, double std, float *out, int threads)
{
    return ng_fill(NG_NORMAL, seed, tensor_id, start, n, mean, std, out, threads);
}

/* out[i] = (float)(lo + (hi - lo) * u(start + i)), i in [0, n). Returns 0 on success. */
int normgen_fill_uniform(uint64_t seed, uint64_t tensor_id, uint64_t start, int64_t n,
                         double lo, double hi, float *out, int threads)
{
    return ng_fill(NG_UNIFORM, seed, tensor_id, start, n, lo, hi, out, threads);
}
