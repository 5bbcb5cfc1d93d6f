// ln_kernels.cu - LayerNorm over long contiguous rows (LayerNorm page,
// POPCORNBENCH transcript "Kimi-K2.6 l1_p40": per row, mean and population
// variance over the normalized extent, y = (x - mean)/sqrt(var + eps) *
// gamma + beta with elementwise gamma/beta).
//
// Statistics.  All partial statistics are (count, mean, M2) triples of
// d = x - K, where the pivot K is an element of the row (the median of its
// first, middle and last elements in the persistent kernel, x[r][0] in the
// split path).
// Shifting by an element of the row keeps the partial sums small when
// |mean| >> std (for x ~ N(1000, 0.01^2) an fp32 sum of raw x would lose the
// variance entirely); d is exact whenever x and K are within a factor of 2.
// Per thread the triple comes from shifted sums (sum d, sum d^2), which a
// pivot inside the bulk of the row keeps well conditioned; triples are
// folded with Chan's pairwise update (Chan, Golub, LeVeque 1979) across the
// warp and the CTA, and across CTAs with the two-pass formula over partials,
// in a fixed order.  The row mean is then K + delta, carried as an
// unevaluated fp32 pair (hi, lo), and the output is
// ((x - hi) - lo) * rstd * gamma + beta.
//
// Persistent path (one CTA per SM, cooperative launch so all CTAs are
// co-resident).  A row is counted in 16-byte units (4 fp32 or 8 bf16
// values); CTA c owns the same column slice of units of every row.  Row
// slices arrive by bulk copy (TMA engine, 32 KB pieces) into two
// shared-memory buffers; the slice of the row being written lives in
// registers (4 registers a unit, bf16 kept packed), and gamma/beta of the
// slice live in tensor memory (TMEM, 4 cells a unit, bf16 kept packed),
// bulk-copied through the row buffers once per launch.  x is read from HBM
// once and stays on chip until y is written; gamma and beta are read from
// HBM once.  Three warp roles run concurrently: warps 1..3 reduce a row's
// statistics as soon as it lands and publish the CTA's triple, warp 0
// merges the triples of all CTAs, warps 4..15 write y.  A row's triples go
// out about two rows before its y is written, which hides the grid-wide
// exchange (several microseconds under full HBM load) behind other rows'
// work.  Before the first y store the apply warps have nothing to write, so
// they reduce rows 0 and 1 together with warps 1..3 (480 threads instead of
// 96); row 0 and gamma are copied first, and beta and row 1 follow into the
// buffers that row 0 and gamma leave.  The pivot's three candidate elements
// travel with each row's bulk copy.
//
// Grid barrier without atomics.  Each CTA publishes its (mean, M2) as two
// 64-bit words, each carrying a 32-bit tag in its high half, in one 16-byte
// record written by a bulk store (cp.async.bulk shared -> global, issued by
// one statistics thread; a generic store would wait behind the CTA's queued
// y stores).  Warp 0 polls the G records of the row with weak L2 loads
// (ld.global.cg, 8 bytes each, which overlap) until every tag matches, so the
// barrier and its data arrive in the same round trip.  It polls after the
// CTA's y stores have been issued: its loads would otherwise queue behind
// them.
// What this relies on: an aligned 8-byte word of the 16-byte record is never
// observed half old and half new by an 8-byte load from L2.  That is a
// property of the hardware (the record is one aligned 16-byte write into one
// L2 sector), not a promise of the PTX memory model, under which these weak
// loads race with the async-proxy store.  Nothing else is needed: each word
// carries its own tag, a word is used only when its tag is the one awaited,
// and a stale word (an older tag) is simply polled again, so no ordering
// between the two words or with other memory is required.  A slot is
// rewritten (4 rows later) only after every CTA has merged the row it held:
// a CTA publishes row q + 4 at its iteration q + 2, which it reaches only
// after merging row q + 2, whose records every CTA publishes only after it
// has merged row q.  Records sit in 4 rotating slots.  Tags count
// rows: row r of a launch is tagged row_base + r + 1, where row_base
// (workspace header) is the number of rows the persistent kernel has already
// processed on this workspace.  A slot therefore only ever holds tags
// smaller than the one awaited, and a zeroed workspace holds tag 0, which is
// never awaited.  row_base is read at kernel start; at its end every CTA
// counts itself in the header, and the last one (which knows that every CTA
// has read row_base) resets the count and advances row_base.
//
// Row groups.  For rows too short for one grid-wide exchange per row to hide
// behind the next rows' traffic, the grid is split into `groups` groups of
// G/groups CTAs: group j takes rows j, j + groups, j + 2 groups, ..., each
// row split over the group's CTAs, and exchanges records only within the
// group.  Slots and buffers follow a group's own row sequence; tags use the
// global row index.  With one group this is the whole grid on every row.  Every wait is
// bounded by %globaltimer: on timeout a CTA records NORM_ERR_TIMEOUT, drains
// its own bulk copies, frees its TMEM and returns without writing its slice
// of the remaining rows (other CTAs may have written theirs).
//
// Split path (any shape): kernel 1 writes one triple per (row, chunk) CTA;
// kernel 2 merges the row's triples and applies, re-reading x.
#include "norm_internal.cuh"
#include <type_traits>

namespace normk {

namespace {

// Warp roles of the persistent kernel: warp 0 coordinates the grid
// barrier, warps 1..3 reduce row statistics from shared memory, warps 4..15
// write y (18 float4 of the slice each, held in registers).
constexpr int LN_THREADS = 512;           // CTA size
constexpr int LN_STATS_WARPS = 3;         // warps 1..3
constexpr int LN_S = 32 * LN_STATS_WARPS; // statistics threads
constexpr int LN_APPLY_WARP0 = 4;         // first apply warp
constexpr int LN_A = LN_THREADS - 32 * LN_APPLY_WARP0; // apply threads (warps 4..15)
constexpr int LN_V = 18;                  // float4 of the slice per apply thread
constexpr int LN_GB = 2;                  // gamma/beta float4 per TMEM load batch
constexpr int LN_NB = LN_V / LN_GB;       // batches per row
constexpr uint32_t LN_TMEM_COLS = 512;    // TMEM columns the CTA allocates (all)
constexpr int LN_TM_COLS = 8 * LN_V;      // TMEM columns of one apply thread: gamma, beta
constexpr uint32_t LN_TM_BETA = 4 * LN_V; // column offset of beta within them
constexpr int LN_SLOTS = 4;               // partial-record slots: reused 4 rows later
constexpr int LN_MAX_GRID = 160;          // CTAs whose records one warp loads at once
// Bytes a bulk copy of a slice moves at once.  With one row group (the whole
// grid on every row) the slices go in 4 KB pieces: measured back to back on
// GB300 at (16, 4194304), 92.9-93.1 us against 94.4 us with 32 KB pieces
// (8 KB 93.7, 16 KB and 128 KB 94.5, 2 KB 99.5 us).  With several row groups
// 32 KB pieces were faster ((256, 262144) in 13 groups: 94.0 us against
// 96.4 us with 4 KB; (64, 1048576) in 4 groups: 91.7 against 92.2 us), and
// small pieces only for the prologue's copies gained less (94.1 us).
constexpr uint32_t LN_BULK_CHUNK = 32768;
constexpr uint32_t LN_BULK_CHUNK_ONE_GROUP = 4096;
constexpr int LN_BAR_APPLIED = 1;         // named barrier of warp 0 and the apply warps
constexpr int LN_BAR_STATS = 2;           // named barrier of the statistics warps
constexpr int LN_BAR_PRO = 3;             // statistics and apply warps (rows 0 and 1)
constexpr int LN_BAR_FILL = 4;            // apply warps (buffers read, gamma/beta to TMEM)
constexpr int LN_PRO_WARPS = LN_THREADS / 32 - 1; // warps that reduce rows 0 and 1
static_assert(LN_V % LN_GB == 0, "whole gamma/beta batches");
static_assert(LN_APPLY_WARP0 % 4 == 0 && LN_A % 128 == 0, "apply warps fill whole TMEM quarters");
// apply warp w sits in TMEM quarter w % 4 and takes column range
// w / 4 - 1 of it, so three of them share a quarter
static_assert((LN_THREADS / 128 - 1) * LN_TM_COLS <= static_cast<int>(LN_TMEM_COLS),
              "gamma/beta of a quarter fit TMEM");

// ---------------------------------------------------------------- persistent path

__device__ __forceinline__ unsigned long long tagged(unsigned tag, float v)
{
    return (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(v);
}

__device__ __forceinline__ unsigned record_tag(unsigned long long w)
{
    return static_cast<unsigned>(w >> 32);
}

__device__ __forceinline__ float record_value(unsigned long long w)
{
    return __uint_as_float(static_cast<unsigned>(w & 0xffffffffull));
}

// Tag of row r's records (never 0, the tag of a zeroed workspace, for the
// first 2^32 - 1 rows processed on a workspace).
__device__ __forceinline__ unsigned row_tag(unsigned row_base, int64_t r)
{
    return row_base + static_cast<unsigned>(r) + 1u;
}

struct GridMerge {
    Moments tot;
    bool ok;
};

// Merge a row's G <= LN_MAX_GRID records (mean, M2 of x - K, all about the
// row's one pivot K), held by warp 0 as w[j][0..1] for CTA lane + 32 j, with
// the two-pass formula over partials:
//   delta = sum_c n_c m_c / N,   M2 = sum_c M2_c + sum_c n_c (m_c - delta)^2,
// with each count n_c known from the partition (qu or qu + 1 units of UE
// elements).  The sums are warp reductions in a fixed order, so every CTA
// computes the same bits; all lanes return the result.
template <int UE>
__device__ __forceinline__ Moments merge_records(const unsigned long long (&w)[LN_MAX_GRID / 32][2], int G,
                                                 unsigned qu, unsigned rem)
{
    constexpr int J = LN_MAX_GRID / 32;
    constexpr float ue = static_cast<float>(UE);
    const int lane = threadIdx.x & 31;
    const float N = ue * (static_cast<float>(qu) * static_cast<float>(G) + static_cast<float>(rem));
    float sm = 0.f; // sum of n_c * m_c
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int i = lane + 32 * j;
        if (i < G) {
            const float n = ue * static_cast<float>(qu + (static_cast<unsigned>(i) < rem ? 1u : 0u));
            sm = fmaf(n, record_value(w[j][0]), sm);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        sm += __shfl_xor_sync(0xffffffffu, sm, o);
    const float delta = __shfl_sync(0xffffffffu, sm, 0) / N;
    float sq = 0.f; // sum of M2_c + n_c (m_c - delta)^2
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int i = lane + 32 * j;
        if (i < G) {
            const float n = ue * static_cast<float>(qu + (static_cast<unsigned>(i) < rem ? 1u : 0u));
            const float dm = record_value(w[j][0]) - delta;
            sq += fmaf(n * dm, dm, record_value(w[j][1]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
    Moments t;
    t.n = N;
    t.mean = delta;
    t.m2 = __shfl_sync(0xffffffffu, sq, 0);
    return t;
}

// Warp 0: read the G records of a row with plain L2 loads (ld.global.cg,
// which overlap) until every tag equals `tag` (bounded by timeout_ns), then
// merge them.
template <int UE>
__device__ __forceinline__ GridMerge poll_and_merge(const unsigned long long *rec, int G, unsigned qu, unsigned rem,
                                                    unsigned tag, uint64_t timeout_ns)
{
    constexpr int J = LN_MAX_GRID / 32;
    const int lane = threadIdx.x & 31;
    GridMerge g;
    g.ok = true;
    uint64_t t0 = 0;
    for (int attempt = 0;; ++attempt) {
        // the words live only inside one attempt, so they stay in registers
        unsigned long long w[J][2];
        unsigned bad = 0;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            // lanes past the last CTA re-read record G-1 (branch-free loads)
            const int i = min(lane + 32 * j, G - 1);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                w[j][e] = ld_cg_u64(rec + 2 * i + e);
                bad |= record_tag(w[j][e]) ^ tag;
            }
        }
        if (__all_sync(0xffffffffu, bad == 0)) {
            g.tot = merge_records<UE>(w, G, qu, rem);
            return g;
        }
        if (attempt == 0)
            t0 = globaltimer_ns();
        else if (__any_sync(0xffffffffu, globaltimer_ns() - t0 > timeout_ns)) {
            g.ok = false;
            return g;
        }
        __nanosleep(32);
    }
}

// Element k of a 16-byte unit of T held in a float4's bits: fp32 component
// k, or bf16 k (the low half of 32-bit word k / 2 for even k), widened.
template <typename T>
__device__ __forceinline__ float unit_elem(const float4 &u, int k)
{
    if constexpr (sizeof(T) == 4) {
        return k == 0 ? u.x : k == 1 ? u.y : k == 2 ? u.z : u.w;
    } else {
        const float wf = (k >> 1) == 0 ? u.x : (k >> 1) == 1 ? u.y : (k >> 1) == 2 ? u.z : u.w;
        const uint32_t wd = __float_as_uint(wf);
        return __uint_as_float((k & 1) ? (wd & 0xffff0000u) : (wd << 16));
    }
}

// The two bf16 of 32-bit word `wf` (held as a float's bits) as an f32x2 pair.
__device__ __forceinline__ float2 bf16_pair(float wf)
{
    const uint32_t wd = __float_as_uint(wf);
    return make_float2(__uint_as_float(wd << 16), __uint_as_float(wd & 0xffff0000u));
}

// Pivot of a row: the median of its first, middle and last elements.  A
// pivot inside the bulk of the row keeps the shifted sums small, and one
// outlier cannot become the pivot.  The three elements arrive by bulk copy
// with the row, each in the 16-byte unit that contains it (row_len is a
// multiple of UE = 16 / sizeof(T), so element i is element i % UE of unit
// i / UE).
template <typename T>
__device__ __forceinline__ float row_pivot(const float4 *piece, int64_t row_len)
{
    constexpr int UE = 16 / static_cast<int>(sizeof(T));
    const int64_t mid = row_len >> 1;
    const float a = unit_elem<T>(piece[0], 0);
    const float b = unit_elem<T>(piece[1], static_cast<int>(mid & (UE - 1)));
    const float c = unit_elem<T>(piece[2], UE - 1);
    return fmaxf(fminf(a, b), fminf(fmaxf(a, b), c));
}

// Shifted sums of d = x - K over units i = pi, pi + np, ... < nu of a row
// slice in shared memory, with four independent accumulator pairs, as this
// thread's (count, mean, M2).  bf16 units (8 values) are shifted by -K a
// 32-bit word at a time (mixed-precision adds) and summed in f32x2 pairs.
template <typename T>
__device__ __forceinline__ Moments slice_moments(const float4 *buf, int nu, int pi, int np, float K)
{
    constexpr int UE = 16 / static_cast<int>(sizeof(T));
    float s1[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
    int i = pi;
    if constexpr (sizeof(T) == 4) {
        for (; i + 3 * np < nu; i += 4 * np) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 v = buf[i + u * np];
                const float a = v.x - K, b = v.y - K, c = v.z - K, d = v.w - K;
                s1[u] += (a + b) + (c + d);
                s2[u] = fmaf(a, a, fmaf(b, b, fmaf(c, c, fmaf(d, d, s2[u]))));
            }
        }
        for (; i < nu; i += np) {
            const float4 v = buf[i];
            const float a = v.x - K, b = v.y - K, c = v.z - K, d = v.w - K;
            s1[0] += (a + b) + (c + d);
            s2[0] = fmaf(a, a, fmaf(b, b, fmaf(c, c, fmaf(d, d, s2[0]))));
        }
    } else {
        const float2 negk = make_float2(-K, -K);
        float2 p1[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        float2 p2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        auto add_unit = [&](const float4 &v, int a) {
            const float2 d0 = bf16x2_add(__float_as_uint(v.x), negk), d1 = bf16x2_add(__float_as_uint(v.y), negk);
            const float2 d2 = bf16x2_add(__float_as_uint(v.z), negk), d3 = bf16x2_add(__float_as_uint(v.w), negk);
            p1[a] = __fadd2_rn(p1[a], __fadd2_rn(__fadd2_rn(d0, d1), __fadd2_rn(d2, d3)));
            p2[a] = __ffma2_rn(d3, d3, __ffma2_rn(d2, d2, __ffma2_rn(d1, d1, __ffma2_rn(d0, d0, p2[a]))));
        };
        for (; i + np < nu; i += 2 * np) {
            add_unit(buf[i], 0);
            add_unit(buf[i + np], 1);
        }
        for (; i < nu; i += np)
            add_unit(buf[i], 0);
        s1[0] = p1[0].x + p1[0].y;
        s1[1] = p1[1].x + p1[1].y;
        s2[0] = p2[0].x + p2[0].y;
        s2[1] = p2[1].x + p2[1].y;
    }
    Moments m = {0.f, 0.f, 0.f};
    const int nv = nu > pi ? (nu - pi + np - 1) / np : 0; // units of this thread
    if (nv > 0) {
        const float S1 = (s1[0] + s1[1]) + (s1[2] + s1[3]);
        const float S2 = (s2[0] + s2[1]) + (s2[2] + s2[3]);
        m.n = static_cast<float>(UE) * static_cast<float>(nv);
        m.mean = S1 / m.n;
        m.m2 = fmaxf(fmaf(-S1, m.mean, S2), 0.f);
    }
    return m;
}

// y of one unit of a LayerNorm row: ((x - hi) - lo) * rstd * gamma + beta.
// fp32: the unit's 4 values, gamma/beta from 4 TMEM cells.  bf16: 8 values,
// gamma/beta 8 packed bf16 in the 4 cells, arithmetic in f32x2 pairs, the
// result packed to bf16 once.  Returns the 16 bytes to store.
template <typename T>
__device__ __forceinline__ float4 ln_unit(const float4 &v, const RowMean &rm, const float4 &g, const float4 &b)
{
    if constexpr (sizeof(T) == 4) {
        return ln_apply4(v, rm, g, b);
    } else {
        const float2 nh = make_float2(-rm.hi, -rm.hi), nl = make_float2(-rm.lo, -rm.lo);
        const float2 r2 = make_float2(rm.rstd, rm.rstd);
        auto word = [&](float xv, float gv, float bv) {
            const float2 t = __fmul2_rn(__fadd2_rn(bf16x2_add(__float_as_uint(xv), nh), nl), r2);
            const float2 o = __ffma2_rn(t, bf16_pair(gv), bf16_pair(bv));
            return __uint_as_float(pack_bf16x2(o.x, o.y));
        };
        return make_float4(word(v.x, g.x, b.x), word(v.y, g.y, b.y), word(v.z, g.z, b.z), word(v.w, g.w, b.w));
    }
}

// One gamma/beta value of the GroupNorm form (read through the read-only
// path; a channel's value is shared by many units).
__device__ __forceinline__ float ldg_param(const float *p)
{
    return __ldg(p);
}

__device__ __forceinline__ float ldg_param(const __nv_bfloat16 *p)
{
    return __bfloat162float(__ldg(p));
}

// y of one unit of the GroupNorm form, all of it in one channel:
// LReLU(((x - hi) - lo) * rstd * g2 + b2) with gamma/beta already doubled.
template <typename T>
__device__ __forceinline__ float4 gn_unit(const float4 &v, const RowMean &rm, float g2, float b2, float slope)
{
    if constexpr (sizeof(T) == 4) {
        float4 o;
        o.x = fmaf(((v.x - rm.hi) - rm.lo) * rm.rstd, g2, b2);
        o.y = fmaf(((v.y - rm.hi) - rm.lo) * rm.rstd, g2, b2);
        o.z = fmaf(((v.z - rm.hi) - rm.lo) * rm.rstd, g2, b2);
        o.w = fmaf(((v.w - rm.hi) - rm.lo) * rm.rstd, g2, b2);
        o.x = o.x > 0.f ? o.x : slope * o.x;
        o.y = o.y > 0.f ? o.y : slope * o.y;
        o.z = o.z > 0.f ? o.z : slope * o.z;
        o.w = o.w > 0.f ? o.w : slope * o.w;
        return o;
    } else {
        const float2 nh = make_float2(-rm.hi, -rm.hi), nl = make_float2(-rm.lo, -rm.lo);
        const float2 r2 = make_float2(rm.rstd, rm.rstd), gg = make_float2(g2, g2), bb = make_float2(b2, b2);
        const float2 s2 = make_float2(slope, slope);
        const bool steep = slope > 1.f;
        auto word = [&](float xv) {
            const float2 t = __ffma2_rn(__fmul2_rn(__fadd2_rn(bf16x2_add(__float_as_uint(xv), nh), nl), r2), gg, bb);
            // LReLU: max(t, slope t) for slope <= 1, min(t, slope t) above
            const float2 u = __fmul2_rn(t, s2);
            const float lo = steep ? fminf(t.x, u.x) : fmaxf(t.x, u.x);
            const float hi = steep ? fminf(t.y, u.y) : fmaxf(t.y, u.y);
            return __uint_as_float(pack_bf16x2(lo, hi));
        };
        return make_float4(word(v.x), word(v.y), word(v.z), word(v.w));
    }
}

// GN: GroupNorm + LeakyReLU + x2 over NCHW segments instead of LayerNorm
// rows: row r is segment r (sample r / G, group r % G) of L = M * S values;
// gamma/beta are per channel (channel g * M + e / S for element e), read
// through L1 per unit (S a multiple of the unit's UE values) instead of held
// in TMEM, and the output is 2 LReLU((x - mean) * rstd * gamma + beta).
// T: float or __nv_bfloat16 (x, y, gamma, beta), fp32 arithmetic.
// ONE: the grid is a single row group (fp32 LayerNorm form only); its slices
// are copied in LN_BULK_CHUNK_ONE_GROUP pieces.
template <typename T, bool GN, bool ONE>
__global__ void __launch_bounds__(LN_THREADS, 1) ln_persistent_kernel(LnParams p, GnPersist gp_)
{
    // A unit is 16 bytes of a row: UE = 4 fp32 or 8 bf16 values.  Slices,
    // buffers, registers (4 a unit) and TMEM cells (4 a unit: gamma/beta of
    // bf16 rows stay packed) are all counted in units.
    constexpr int UE = 16 / static_cast<int>(sizeof(T));
    extern __shared__ __align__(128) float4 ln_smem[];
    __shared__ __align__(8) uint64_t bar_x[2];
    __shared__ __align__(8) uint64_t bar_g, bar_b; // gamma into buffer 1, beta into buffer 0
    __shared__ Moments red[2][LN_PRO_WARPS];            // per-warp triples, by row parity
    __shared__ __align__(16) unsigned long long rec_out[2][2]; // this CTA's record, by row parity
    __shared__ float4 piv_in[2][3];                     // a row's pivot candidates, by row parity
    __shared__ float piv_k[2];                          // a row's pivot, by row parity
    __shared__ RowMean row_mean[2];                     // merged statistics, by row parity
    __shared__ unsigned row_base_s;
    __shared__ uint32_t tmem_base_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int NG = p.groups;         // row groups
    const int Gk = G / NG;           // CTAs per group
    const int grp = cta / Gk;        // this CTA's group
    const int crank = cta - grp * Gk; // its rank in the group
    // The group's rows: local row t is row grp + t * NG of the launch.
    const int64_t R = p.rows > grp ? (p.rows - grp + NG - 1) / NG : 0;
    auto grow = [&](int64_t t) { return grp + t * NG; };
    // units per row by a shift: a signed 64-bit division by UE (an exact one,
    // row_len being a multiple of UE) cost 0.4-0.5 us a launch of
    // (16, 4194304) fp32 in instructions the compiler recomputes in the loops
    constexpr int UE_SHIFT = UE == 4 ? 2 : 3;
    const int64_t Lu = p.row_len >> UE_SHIFT;
    // CTA rank c owns nu = qu (+1 for the first rem ranks) units of every row
    // of its group, starting at f0; the merge recomputes every rank's count
    // the same way.
    const unsigned qu = static_cast<unsigned>(Lu / Gk), rem = static_cast<unsigned>(Lu % Gk);
    const int64_t f0 = static_cast<int64_t>(crank) * qu + min(static_cast<unsigned>(crank), rem);
    const int nu = static_cast<int>(qu + (static_cast<unsigned>(crank) < rem ? 1u : 0u));
    const float4 *x4 = reinterpret_cast<const float4 *>(p.x);
    float4 *y4 = reinterpret_cast<float4 *>(p.y);
    const float4 *g4 = reinterpret_cast<const float4 *>(p.gamma);
    const float4 *b4 = reinterpret_cast<const float4 *>(p.beta);
    unsigned long long *records = reinterpret_cast<unsigned long long *>(p.part);
    const int buf_u = (p.max_n4 + 7) & ~7;

    const uint64_t pol_stream = policy_evict_first();
    // bulk copy of `bytes` from src to dst on bar, in pieces (see
    // LN_BULK_CHUNK)
    auto copy_in = [&](float4 *dst, const float4 *src, uint32_t bytes, uint64_t *bar) {
        constexpr uint32_t piece = ONE ? LN_BULK_CHUNK_ONE_GROUP : LN_BULK_CHUNK;
        for (uint32_t off = 0; off < bytes; off += piece)
            bulk_g2s(dst + off / 16, src + off / 16, (bytes - off < piece) ? (bytes - off) : piece, bar, pol_stream);
    };
    // Waits for this CTA's own bulk copies after a failure (drains) use at
    // least 100 ms, whatever the configured limit: a copy always completes
    // in microseconds, and the CTA must not exit while one still writes its
    // shared memory.
    const uint64_t drain_ns = p.timeout_ns > 100000000ull ? p.timeout_ns : 100000000ull;

    // The CTA holds all 512 TMEM columns (it is alone on its SM: its 512
    // threads at 128 registers take the whole register file).
    if (!GN && warp == 0)
        tmem_alloc(&tmem_base_s, LN_TMEM_COLS);
    if (tid == 0) {
        mbar_init(&bar_x[0], 1);
        mbar_init(&bar_x[1], 1);
        mbar_init(&bar_g, 1);
        mbar_init(&bar_b, 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        row_base_s = ld_relaxed_gpu_u32(&p.sync->row_base);
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const unsigned row_base = row_base_s;
    const uint32_t tmem_base = GN ? 0u : tmem_base_s;
    bool aborted = false;

    // Row q's slice, plus the three 16-byte pieces of the row that hold its
    // pivot candidates, all on bar_x[q & 1] (row q lives in buffer q & 1).
    auto issue_x = [&](int64_t q) {
        uint64_t *bar = &bar_x[q & 1];
        const uint32_t bytes = static_cast<uint32_t>(nu) * 16u;
        mbar_arrive_expect_tx(bar, bytes + 48u);
        const float4 *row = x4 + grow(q) * Lu;
        bulk_g2s(&piv_in[q & 1][0], row, 16u, bar, pol_stream);
        bulk_g2s(&piv_in[q & 1][1], row + ((p.row_len >> 1) >> UE_SHIFT), 16u, bar, pol_stream);
        bulk_g2s(&piv_in[q & 1][2], row + (Lu - 1), 16u, bar, pol_stream);
        const float4 *src = row + f0;
        float4 *dst = ln_smem + (q & 1) * buf_u;
        copy_in(dst, src, bytes, bar);
    };
    auto x_parity = [](int64_t q) { return static_cast<uint32_t>((q >> 1) & 1); };

    // Iteration r (-2 <= r < R) starts with a block-wide barrier that is
    // also the abort vote (__syncthreads_or).  By then warp 0 has merged row
    // r.  During it:
    //   warps 1..3    reduce row r+2 from its buffer (it lands meanwhile) and
    //                 publish the CTA's triple of it at once;
    //   warps 4..15   write y of row r, move row r+1 from its buffer into
    //                 registers, and meet warp 0 at barrier LN_BAR_APPLIED;
    //                 then warp 4 refills that buffer with row r+3;
    //   warp 0        after LN_BAR_APPLIED, merges row r+1, whose triples
    //                 every CTA published during the previous iteration.
    // A row's triples are published about two iterations before its y is
    // written, so the grid-wide exchange has that long to complete, and the
    // reduction of a row overlaps the writing of an earlier one.
    // Prologue (r = -2, -1): no y is written yet, so the apply warps reduce
    // rows 0 and 1 together with the statistics warps (15 warps instead of
    // 3; LN_BAR_PRO).  Row 0 (buffer 0) and gamma (buffer 1) are copied at the
    // start.  As soon as row 0 is reduced the apply warps move it into their
    // registers, which frees buffer 0 for beta; gamma goes from buffer 1 to
    // TMEM, which frees buffer 1 for row 1; then beta goes to TMEM.  So row 0
    // crosses the grid while gamma, beta and row 1 are still arriving.
    // (every group has a row: the host never makes more groups than rows)
    if (R == 0) {
        // nothing to do
    } else if (warp == 0) {
        // ------------------------------------------------ coordinator
        bool fail = false; // the merge of the previous row gave up
        for (int64_t r = -2; r < R; ++r) {
            if (__syncthreads_or(fail ? 1 : 0)) {
                aborted = true;
                break;
            }
            const int64_t q = r + 1; // the row merged now
            // Poll once the apply warps have issued their y stores: loads
            // issued while those stores queue would wait behind them.
            bar_sync_named(LN_BAR_APPLIED, LN_A + 32);
            if (q >= 0 && q < R) {
                const GridMerge gm =
                    poll_and_merge<UE>(records + (static_cast<int64_t>(q % LN_SLOTS) * G + grp * Gk) * 2, Gk, qu, rem,
                                   row_tag(row_base, grow(q)) + p.tag_skew, p.timeout_ns);
                if (!gm.ok) {
                    fail = true;
                    if (lane == 0)
                        record_error(p.err, NORM_ERR_TIMEOUT);
                } else if (lane == 0) {
                    row_mean[q & 1] = finish_row(piv_k[q & 1], gm.tot, p.eps);
                }
            }
        }
    } else if (warp < LN_APPLY_WARP0) {
        // ------------------------------------------------ statistics warps 1..3
        const int st = tid - 32;
        bool fail = false; // row q's copy did not land in time
        for (int64_t r = -2; r < R; ++r) {
            if (__syncthreads_or(fail ? 1 : 0)) {
                aborted = true;
                break;
            }
            const int64_t q = r + 2; // the row reduced and published now
            if (q >= R)
                continue;
            // rows 0 and 1 are reduced by the apply warps too
            const bool pro = q < 2;
            const int np = pro ? 32 * LN_PRO_WARPS : LN_S;
            fail = !mbar_wait_bounded(&bar_x[q & 1], x_parity(q), p.timeout_ns);
            const float K = fail ? 0.f : row_pivot<T>(piv_in[q & 1], p.row_len);
            Moments m = {0.f, 0.f, 0.f};
            if (!fail)
                m = slice_moments<T>(ln_smem + (q & 1) * buf_u, nu, st, np, K);
            m = warp_merge(m);
            if (lane == 0)
                red[q & 1][warp - 1] = m;
            if (pro)
                bar_sync_named(LN_BAR_PRO, 32 * LN_PRO_WARPS);
            else
                bar_sync_named(LN_BAR_STATS, LN_S);
            if (warp == 1) {
                // The CTA's triple of row q goes out now as a 16-byte bulk
                // store: a plain store would stall this warp until the
                // CTA's y stores ahead of it drain.
                Moments c = {0.f, 0.f, 0.f};
                if (lane < (pro ? LN_PRO_WARPS : LN_STATS_WARPS))
                    c = red[q & 1][lane];
                c = warp_merge(c);
                if (lane == 0 && !fail) {
                    piv_k[q & 1] = K;
                    const unsigned tag = row_tag(row_base, grow(q));
                    // the store of row q - 2 has read its source
                    bulk_wait_read_all();
                    rec_out[q & 1][0] = tagged(tag, c.mean);
                    rec_out[q & 1][1] = tagged(tag, c.m2);
                    fence_proxy_async_smem();
                    bulk_s2g(records + (static_cast<int64_t>(q % LN_SLOTS) * G + cta) * 2, rec_out[q & 1], 16);
                    bulk_commit();
                }
            }
        }
        // the last record has left shared memory
        if (st == 0)
            bulk_wait_all();
    } else {
        // ------------------------------------------------ apply warps 4..15
        const int at = tid - 32 * LN_APPLY_WARP0;
        const int pt = tid - 32; // index among the warps that reduce rows 0 and 1
        // Thread 32 * LN_APPLY_WARP0 issues the bulk copies.  It tracks the
        // rows it issued (rows < issued) and those whose completion it
        // observed (rows < waited), and the same for gamma and beta, so that
        // an early exit can drain them.
        const bool issuer = at == 0;
        int64_t issued = 0, waited = 0;
        bool g_out = false, b_out = false; // gamma / beta copy issued and not seen complete
        bool fail = false; // a copy the prologue waits for did not land in time
        // gamma or beta of the slice (h = 0, 1) into buffer 1 or 0, on bar
        auto issue_param = [&](const float4 *src, int buf, uint64_t *bar) {
            const uint32_t bytes = src ? static_cast<uint32_t>(nu) * 16u : 0u;
            mbar_arrive_expect_tx(bar, bytes);
            float4 *dst = ln_smem + buf * buf_u;
            copy_in(dst, src + f0, bytes, bar);
        };
        if (issuer) {
            issue_x(0);
            issued = 1;
            if (GN) {
                // no gamma/beta to stage: row 1 goes to buffer 1 at once
                if (R > 1) {
                    issue_x(1);
                    issued = 2;
                }
            } else {
                issue_param(g4, 1, &bar_g);
                g_out = true;
            }
        }
        // This thread's TMEM cells: lane 32*(warp % 4) + lane of its warp's
        // quarter, LN_TM_COLS columns from (warp / 4 - 1) * LN_TM_COLS:
        // gamma of its k-th float4 at column 4k, beta at LN_TM_BETA + 4k.
        const uint32_t tm = tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16) +
                            static_cast<uint32_t>((warp / 4 - 1) * LN_TM_COLS);
        // Help reduce prologue row q (0 or 1) from its buffer: this thread's
        // share of the 15-warp partition, merged over the warp, to red[].
        auto help_reduce = [&](int64_t q) {
            const bool ok = mbar_wait_bounded(&bar_x[q & 1], x_parity(q), p.timeout_ns);
            fail = fail || !ok;
            if (ok && issuer)
                waited = q + 1;
            Moments m = {0.f, 0.f, 0.f};
            if (ok)
                m = slice_moments<T>(ln_smem + (q & 1) * buf_u, nu, pt, 32 * LN_PRO_WARPS,
                                     row_pivot<T>(piv_in[q & 1], p.row_len));
            m = warp_merge(m);
            if (lane == 0)
                red[q & 1][warp - 1] = m;
            bar_sync_named(LN_BAR_PRO, 32 * LN_PRO_WARPS);
        };
        // gamma or beta (wait on bar, then buffer buf -> this thread's TMEM
        // columns from col0; the unit d where the parameter is absent)
        auto fill_tmem = [&](const float4 *src, int buf, uint64_t *bar, uint32_t col0, float4 d) {
            const bool ok = mbar_wait_bounded(bar, 0, p.timeout_ns);
            fail = fail || !ok;
            const float4 *b = ln_smem + buf * buf_u;
            __syncwarp();
#pragma unroll
            for (int k = 0; k < LN_V; k += 2) {
                float4 a0, a1;
                const int i0 = at + k * LN_A, i1 = at + (k + 1) * LN_A;
                a0 = (src && ok && i0 < nu) ? b[i0] : d;
                a1 = (src && ok && i1 < nu) ? b[i1] : d;
                tmem_st4(tm + col0 + static_cast<uint32_t>(4 * k), a0);
                tmem_st4(tm + col0 + static_cast<uint32_t>(4 * (k + 1)), a1);
            }
            tmem_wait_st();
            return ok;
        };
        float4 v[LN_V]; // this thread's part of the slice of row r
        for (int64_t r = -2; r < R; ++r) {
            if (__syncthreads_or(fail ? 1 : 0)) {
                aborted = true;
                break;
            }
            if (GN && r == -2) {
                // row 0: reduce it with the statistics warps, then hold it in
                // registers (buffer 0 takes row 2 at r = -1)
                help_reduce(0);
#pragma unroll
                for (int k = 0; k < LN_V; ++k) {
                    const int i = at + k * LN_A;
                    v[k] = (i < nu) ? ln_smem[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                __syncwarp();
            } else if (r == -2) {
                // row 0: reduce it with the statistics warps, then hold it in
                // registers, so its buffer can take beta
                help_reduce(0);
#pragma unroll
                for (int k = 0; k < LN_V; ++k) {
                    const int i = at + k * LN_A;
                    v[k] = (i < nu) ? ln_smem[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                // every apply thread has read buffer 0 (the statistics warps
                // finished with it at LN_BAR_PRO)
                bar_sync_named(LN_BAR_FILL, LN_A);
                if (issuer && !fail) {
                    fence_proxy_async_smem();
                    issue_param(b4, 0, &bar_b);
                    b_out = true;
                }
                // gamma: buffer 1 -> TMEM, then row 1 into buffer 1
                // an absent gamma is 1: four fp32 ones, or eight bf16 ones
                const float one = sizeof(T) == 4 ? 1.f : __uint_as_float(0x3f803f80u);
                const bool g_ok = fill_tmem(g4, 1, &bar_g, 0u, make_float4(one, one, one, one));
                if (issuer && g_ok)
                    g_out = false;
                bar_sync_named(LN_BAR_FILL, LN_A);
                if (issuer && !fail && R > 1) {
                    fence_proxy_async_smem();
                    issue_x(1);
                    issued = 2;
                }
                // beta: buffer 0 -> TMEM (buffer 0 takes row 2 at r = -1)
                const bool b_ok = fill_tmem(b4, 0, &bar_b, LN_TM_BETA, make_float4(0.f, 0.f, 0.f, 0.f));
                if (issuer && b_ok)
                    b_out = false;
                bar_sync_named(LN_BAR_FILL, LN_A);
            }
            if (GN && r >= 0) {
                // y of segment r from registers: 2 LReLU(d * rstd * gamma_c +
                // beta_c), gamma/beta doubled (LReLU is positively homogeneous
                // and doubling is exact).  Unit k of this thread starts at
                // element e_k = e_0 + UE LN_A k of the segment; its channel is
                // e_k / S within the group, tracked incrementally.
                const RowMean rm = row_mean[r & 1];
                const int64_t gr = grow(r);
                const int64_t cbase = small_mod(gr, gp_.G) * gp_.M;
                float4 *yr = y4 + gr * Lu + f0;
                constexpr uint32_t step = static_cast<uint32_t>(UE) * LN_A;
                const uint32_t S = gp_.S, e0 = static_cast<uint32_t>(UE) * static_cast<uint32_t>(f0 + at);
                uint32_t cq = e0 / S, rq = e0 - cq * S;
                const T *gp = p.gamma ? static_cast<const T *>(p.gamma) + cbase : nullptr;
                const T *bp = p.beta ? static_cast<const T *>(p.beta) + cbase : nullptr;
#pragma unroll
                for (int k = 0; k < LN_V; ++k) {
                    const int i = at + k * LN_A;
                    if (i < nu) {
                        const float gv = gp ? ldg_param(gp + cq) : 1.f, bv = bp ? ldg_param(bp + cq) : 0.f;
                        st_stream_f4(yr + i, gn_unit<T>(v[k], rm, gv + gv, bv + bv, gp_.slope), pol_stream);
                    }
                    // next unit: UE LN_A elements on
                    rq += step;
                    if (S >= step) {
                        if (rq >= S) {
                            rq -= S;
                            ++cq;
                        }
                    } else {
                        const uint32_t e = e0 + step * static_cast<uint32_t>(k + 1);
                        cq = e / S;
                        rq = e - cq * S;
                    }
                }
            } else if (r >= 0) {
                // y of row r from registers, gamma/beta from TMEM in batches
                // of LN_GB float4
                const RowMean rm = row_mean[r & 1];
                float4 *yr = y4 + grow(r) * Lu + f0;
#pragma unroll
                for (int bt = 0; bt < LN_NB; ++bt) {
                    float4 g[LN_GB], bb[LN_GB];
                    // tcgen05 loads and waits are warp-collective: reconverge
                    // after the divergent stores first
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < LN_GB; ++j) {
                        const uint32_t c = static_cast<uint32_t>(4 * (bt * LN_GB + j));
                        g[j] = tmem_ld4(tm + c);
                        bb[j] = tmem_ld4(tm + LN_TM_BETA + c);
                    }
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < LN_GB; ++j) {
                        tmem_pin(g[j]);
                        tmem_pin(bb[j]);
                    }
#pragma unroll
                    for (int j = 0; j < LN_GB; ++j) {
                        const int k = bt * LN_GB + j;
                        const int i = at + k * LN_A;
                        if (i < nu)
                            st_stream_f4(yr + i, ln_unit<T>(v[k], rm, g[j], bb[j]), pol_stream);
                    }
                }
            }
            const int64_t q = r + 1; // the row moved into registers now (row 0 was at r = -2)
            if (q >= 1 && q < R) {
                // row q landed before it was reduced (an iteration ago); the
                // issuer's wait returns at once and lets it account for the copy
                if (issuer && mbar_wait_bounded(&bar_x[q & 1], x_parity(q), drain_ns))
                    waited = q + 1;
                const float4 *buf = ln_smem + (q & 1) * buf_u;
#pragma unroll
                for (int k = 0; k < LN_V; ++k) {
                    const int i = at + k * LN_A;
                    v[k] = (i < nu) ? buf[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            __syncwarp();
            bar_sync_named(LN_BAR_APPLIED, LN_A + 32);
            // buffer q & 1 and its pivot pieces are free (row q was reduced
            // an iteration ago, and beta left buffer 0 at r = -2): refill them
            // with row q + 2
            if (issuer && q >= 0 && q + 2 < R) {
                fence_proxy_async_smem();
                issue_x(q + 2);
                issued = q + 3;
            }
            // r = -1: help reduce row 1 while warp 0 merges row 0
            if (r == -1 && R > 1)
                help_reduce(1);
        }
        // Drain: never leave a bulk copy in flight into shared memory.
        if (issuer) {
            for (int64_t qq = waited; qq < issued; ++qq) {
                if (!mbar_wait_bounded(&bar_x[qq & 1], x_parity(qq), drain_ns))
                    record_error(p.err, NORM_ERR_TIMEOUT);
            }
            if (g_out && !mbar_wait_bounded(&bar_g, 0, drain_ns))
                record_error(p.err, NORM_ERR_TIMEOUT);
            if (b_out && !mbar_wait_bounded(&bar_b, 0, drain_ns))
                record_error(p.err, NORM_ERR_TIMEOUT);
        }
    }
    // Whichever role's wait gave up, the vote ended every role's loop: one
    // record of the failure for the CTA.
    if (aborted && tid == 0)
        record_error(p.err, NORM_ERR_TIMEOUT);
    // Every TMEM access of every thread is complete before warp 0 frees it.
    tmem_fence_before_sync();
    __syncthreads();
    // This CTA is done with row_base; the last CTA of the launch advances it
    // by the launch's rows (and resets the count for the next launch).
    if (tid == 0) {
        const unsigned seen = atomicAdd(&p.sync->done, 1u);
        if (seen == static_cast<unsigned>(G) - 1u) {
            st_relaxed_gpu_u32(&p.sync->done, 0u);
            st_relaxed_gpu_u32(&p.sync->row_base, row_base + static_cast<unsigned>(p.rows));
        }
    }
    if (!GN && warp == 0) {
        tmem_fence_after_sync();
        tmem_dealloc(tmem_base, LN_TMEM_COLS);
    }
}

// ---------------------------------------------------------------- row path
//
// Rows of at most 512 threads x 8 4-element vectors (16,384 elements), length a
// multiple of 4, 16-byte aligned: one CTA per row at a time (grid-stride over rows),
// the row in registers, so x is read from HBM once and there is no
// workspace and a single launch.  Mean and M2 are the exact two-pass
// definition over the registers, about the pivot K = x[r][0]:
//   delta = sum(x - K) / L, mean = K + delta (an fp32 pair), M2 = sum((x -
//   mean)^2).
// Several CTAs per SM keep several rows in flight.

// NT threads a CTA, V 4-element vectors a thread.  The bf16 forms with
// packed rows (V >= 16) and with 4 vectors a thread are held to 1,024
// threads an SM's worth of registers (63-64 a thread: at NT = 64, 16 CTAs an
// SM instead of 14 at the 72 the packed form takes unbounded).  Measured
// back to back on GB300: bf16 (16384, 4096) 47.7 -> 45.1 us, (8192, 8192)
// 48.0 -> 45.4 us, (16384, 8192) 89.3 -> 86.2 us, (131072, 512) 58.4 ->
// 54.9 us; a bound of 1,152 threads (56 registers) gave 46.7, 47.2 and 89.0
// us, tighter bounds spilled, and the same bound on 8 vectors a thread was
// slower ((65536, 1024) 45.7 -> 47.5 us).
template <typename T, int NT, int V>
__global__ void __launch_bounds__(NT, (sizeof(T) == 2 && (V >= 16 || V == 4)) ? 1024 / NT : 1)
    ln_rows_kernel(LnParams p)
{
    pdl_begin();
    __shared__ float red[2][NT / 32];
    const int tid = threadIdx.x;
    const int64_t L4 = p.row_len >> 2; // 4-element vectors per row
    const float invL = 1.f / static_cast<float>(p.row_len); // the means below are products, not divisions
    const T *x = static_cast<const T *>(p.x);
    T *y = static_cast<T *>(p.y);
    const T *gm = static_cast<const T *>(p.gamma);
    const T *bt = static_cast<const T *>(p.beta);
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    // small rows hold gamma/beta in registers across rows; large rows load
    // them (L2-resident) when applying
    constexpr bool KEEP_GB = V <= 4;
    float4 gk[KEEP_GB ? V : 1], bk[KEEP_GB ? V : 1];
    if (KEEP_GB) {
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t i = tid + k * NT;
            gk[k] = (gm && i < L4) ? Io<T>::ld4_ro(gm + 4 * i, pol_keep) : make_float4(1.f, 1.f, 1.f, 1.f);
            bk[k] = (bt && i < L4) ? Io<T>::ld4_ro(bt + 4 * i, pol_keep) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    // fp32 rows, and bf16 rows of at most 8 vectors a thread, are held as
    // d = x - K in f32x2 pairs.  bf16 rows of 16 vectors a thread are held
    // packed as loaded (two registers a vector, so a thread keeps twice the
    // bytes in flight that widened values would allow) and widened in each
    // pass; measured faster for rows of 4,096 and 8,192 values, slower for
    // shorter rows, where it adds the widening without adding bytes in flight.
    constexpr bool RAW = sizeof(T) == 2 && V >= 16;
    for (int64_t r = blockIdx.x; r < p.rows; r += gridDim.x) {
        const T *xr = x + r * p.row_len;
        float2 vl[RAW ? 1 : V], vh[RAW ? 1 : V];
        uint2 raw[RAW ? V : 1];
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t i = tid + k * NT;
            if constexpr (RAW) {
                raw[k] = make_uint2(0u, 0u);
                if (i < L4)
                    asm("ld.global.L1::no_allocate.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
                        : "=r"(raw[k].x), "=r"(raw[k].y)
                        : "l"(xr + 4 * i), "l"(pol_stream));
            } else {
                const float4 t =
                    i < L4 ? Io<T>::ld4_stream(xr + 4 * i, pol_stream) : make_float4(0.f, 0.f, 0.f, 0.f);
                vl[k] = make_float2(t.x, t.y);
                vh[k] = make_float2(t.z, t.w);
            }
        }
        // the vector's pairs widened and shifted by off (bf16), or the held
        // pairs plus off (fp32, already d = x - K)
        auto pair = [&](int k, float2 off, float2 &l, float2 &h) {
            if constexpr (RAW) {
                // a shift and a mask a pair: measured faster here than the
                // mixed-precision adds of the other kernels (47.5 against
                // 50.2 us at (16384, 4096))
                l = __fadd2_rn(make_float2(__uint_as_float(raw[k].x << 16), __uint_as_float(raw[k].x & 0xffff0000u)),
                               off);
                h = __fadd2_rn(make_float2(__uint_as_float(raw[k].y << 16), __uint_as_float(raw[k].y & 0xffff0000u)),
                               off);
            } else {
                l = __fadd2_rn(vl[k], off);
                h = __fadd2_rn(vh[k], off);
            }
        };
        // every thread reads the pivot before any thread of the CTA stores
        // (the block sums below are barriers), so y == x is safe
        const float K = Io<T>::ld1(xr);
        const float2 negk = make_float2(-K, -K), zero2 = make_float2(0.f, 0.f);
        // from here on the fp32 pairs hold d = x - K (zero outside the row)
        float2 sl = zero2, sh = zero2;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            if (tid + k * NT < L4) {
                float2 l, h;
                pair(k, negk, l, h);
                if constexpr (!RAW) {
                    vl[k] = l;
                    vh[k] = h;
                }
                sl = __fadd2_rn(sl, l);
                sh = __fadd2_rn(sh, h);
            }
        }
        float s = (sl.x + sl.y) + (sh.x + sh.y);
        s = block_sum<NT>(s, red[0]);
        const float mean_d = s * invL;
        const float2 nm = make_float2(-mean_d, -mean_d);
        // deviations from the mean: d - mean_d (fp32), or x - (K + mean_d)
        // with the centre rounded once (bf16; its offset from the exact
        // centre adds at most L * ulp(K)^2 / 4 to M2)
        const float2 nc = RAW ? make_float2(-(K + mean_d), -(K + mean_d)) : nm;
        float2 ql = zero2, qh = zero2;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            if (tid + k * NT < L4) {
                float2 el, eh;
                pair(k, nc, el, eh);
                ql = __ffma2_rn(el, el, ql);
                qh = __ffma2_rn(eh, eh, qh);
            }
        }
        float q = (ql.x + ql.y) + (qh.x + qh.y);
        q = block_sum<NT>(q, red[1]);
        const float rstd = rsqrtf(fmaxf(q * invL, 0.f) + p.eps);
        const float2 r2 = make_float2(rstd, rstd);
        T *yr = y + r * p.row_len;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t i = tid + k * NT;
            if (i < L4) {
                float4 g, b;
                if (KEEP_GB) {
                    g = gk[k];
                    b = bk[k];
                } else {
                    g = gm ? Io<T>::ld4_param(gm + 4 * i) : make_float4(1.f, 1.f, 1.f, 1.f);
                    b = bt ? Io<T>::ld4_param(bt + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                // y = (d - mean_d) * rstd * g + b = d * a + c, a = rstd * g,
                // c = b - mean_d * a
                float2 dl, dh;
                pair(k, RAW ? negk : zero2, dl, dh);
                const float2 al = __fmul2_rn(make_float2(g.x, g.y), r2), ah = __fmul2_rn(make_float2(g.z, g.w), r2);
                const float2 ol = __ffma2_rn(dl, al, __ffma2_rn(nm, al, make_float2(b.x, b.y)));
                const float2 oh = __ffma2_rn(dh, ah, __ffma2_rn(nm, ah, make_float2(b.z, b.w)));
                Io<T>::st4_stream(yr + 4 * i, make_float4(ol.x, ol.y, oh.x, oh.y), pol_stream);
            }
        }
    }
}

// ---------------------------------------------------------------- split path

constexpr int LS_T = 256;

// One triple per (chunk p, row r) CTA.  Vector form: each thread keeps four
// 4-element loads in flight and accumulates the shifted sums sum d and
// sum d^2 of d = x - K, which the pivot (an element of the row) keeps well
// conditioned, then turns them into its (n, mean, M2); scalar form is
// Welford.  The threads' triples are merged with Chan's update.
template <typename T, bool VEC>
__global__ void __launch_bounds__(LS_T) ln_split_stats_kernel(LnParams p)
{
    pdl_begin();
    __shared__ Moments red[LS_T / 32];
    const int P = p.parts;
    const T *x = static_cast<const T *>(p.x);
    for (int64_t r = blockIdx.y; r < p.rows; r += gridDim.y) {
        const int pc = blockIdx.x;
        const T *xr = x + r * p.row_len;
        const float K = Io<T>::ld1(xr);
        const int64_t lo = static_cast<int64_t>(pc) * p.chunk;
        const int64_t hi = (lo + p.chunk < p.row_len) ? lo + p.chunk : p.row_len;
        Moments m = {0.f, 0.f, 0.f};
        if (VEC) {
            // x stays in L2 for the apply kernel's re-read where it fits
            const uint64_t pol = policy_evict_last();
            float s1 = 0.f, s2 = 0.f, cnt = 0.f;
            auto add = [&](const float4 &q) {
                const float a = q.x - K, b = q.y - K, c = q.z - K, d = q.w - K;
                s1 += (a + b) + (c + d);
                s2 += (a * a + b * b) + (c * c + d * d);
                cnt += 4.f;
            };
            int64_t i = lo / 4 + threadIdx.x;
            const int64_t e4 = hi / 4;
            for (; i + 3 * LS_T < e4; i += 4 * LS_T) {
                float4 q[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    q[u] = Io<T>::ld4_stream(xr + 4 * (i + u * LS_T), pol);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    add(q[u]);
            }
            for (; i < e4; i += LS_T)
                add(Io<T>::ld4_stream(xr + 4 * i, pol));
            if (cnt > 0.f) {
                m.n = cnt;
                m.mean = s1 / cnt;
                m.m2 = fmaxf(s2 - s1 * m.mean, 0.f);
            }
        } else {
            for (int64_t i = lo + threadIdx.x; i < hi; i += LS_T) {
                const float d = Io<T>::ld1(xr + i) - K;
                m.n += 1.f;
                const float delta = d - m.mean;
                m.mean += delta / m.n;
                m.m2 = fmaf(delta, d - m.mean, m.m2);
            }
        }
        const Moments cm = cta_merge<LS_T>(m, red);
        // The pivot travels with the partial: with y == x, the apply kernel
        // may already have overwritten x[r][0] when another CTA needs it.
        if (threadIdx.x == 0)
            p.part[r * P + pc] = make_float4(cm.n, cm.mean, cm.m2, K);
        __syncthreads();
    }
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(LS_T) ln_split_apply_kernel(LnParams p)
{
    pdl_begin();
    __shared__ RowMean row_mean;
    const int P = p.parts;
    const T *x = static_cast<const T *>(p.x);
    T *y = static_cast<T *>(p.y);
    const T *gm = static_cast<const T *>(p.gamma);
    const T *bt = static_cast<const T *>(p.beta);
    // Rows and chunks in the reverse of the statistics kernel's order: the
    // most recently read part of x is the likeliest still in L2.
    for (int64_t rr = blockIdx.y; rr < p.rows; rr += gridDim.y) {
        const int64_t r = p.rows - 1 - rr;
        const int pc = P - 1 - static_cast<int>(blockIdx.x);
        const T *xr = x + r * p.row_len;
        T *yr = y + r * p.row_len;
        if (threadIdx.x < 32) {
            const float K = ld_l2_f4(p.part + r * P).w;
            const Moments tot = merge_partials_warp(p.part + r * P, P, K);
            if (threadIdx.x == 0)
                row_mean = finish_row(K, tot, p.eps);
        }
        __syncthreads();
        const RowMean rm = row_mean;
        const int64_t lo = static_cast<int64_t>(pc) * p.chunk;
        const int64_t hi = (lo + p.chunk < p.row_len) ? lo + p.chunk : p.row_len;
        if (VEC) {
            const uint64_t pol = policy_evict_first();
            const uint64_t pol_gb = policy_evict_last();
            auto one = [&](int64_t i, const float4 &q) {
                const float4 g = gm ? Io<T>::ld4_ro(gm + 4 * i, pol_gb) : make_float4(1.f, 1.f, 1.f, 1.f);
                const float4 bb = bt ? Io<T>::ld4_ro(bt + 4 * i, pol_gb) : make_float4(0.f, 0.f, 0.f, 0.f);
                Io<T>::st4_stream(yr + 4 * i, ln_apply4(q, rm, g, bb), pol);
            };
            int64_t i = lo / 4 + threadIdx.x;
            const int64_t e4 = hi / 4;
            // four loads of x in flight per thread
            for (; i + 3 * LS_T < e4; i += 4 * LS_T) {
                float4 q[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    q[u] = Io<T>::ld4_stream(xr + 4 * (i + u * LS_T), pol);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    one(i + u * LS_T, q[u]);
            }
            for (; i < e4; i += LS_T)
                one(i, Io<T>::ld4_stream(xr + 4 * i, pol));
        } else {
            for (int64_t i = lo + threadIdx.x; i < hi; i += LS_T) {
                const float g = gm ? Io<T>::ld1(gm + i) : 1.f;
                const float bb = bt ? Io<T>::ld1(bt + i) : 0.f;
                Io<T>::st1(yr + i, fmaf(((Io<T>::ld1(xr + i) - rm.hi) - rm.lo) * rm.rstd, g, bb));
            }
        }
        __syncthreads();
    }
}

} // namespace

LnPersistentConfig ln_persistent_config()
{
    return LnPersistentConfig{LN_THREADS, LN_A, LN_V, LN_SLOTS * 16, LN_MAX_GRID};
}

namespace {

// The persistent kernel's forms: fp32 and bf16 LayerNorm (fp32 also with a
// single row group) and GroupNorm.
const void *const kPersistentForms[] = {reinterpret_cast<const void *>(ln_persistent_kernel<float, false, false>),
                                        reinterpret_cast<const void *>(ln_persistent_kernel<float, false, true>),
                                        reinterpret_cast<const void *>(ln_persistent_kernel<float, true, false>),
                                        reinterpret_cast<const void *>(ln_persistent_kernel<__nv_bfloat16, false, false>),
                                        reinterpret_cast<const void *>(ln_persistent_kernel<__nv_bfloat16, true, false>)};

const void *persistent_form(bool bf16, bool gn, bool one_group)
{
    if (bf16)
        return gn ? kPersistentForms[4] : kPersistentForms[3];
    return gn ? kPersistentForms[2] : one_group ? kPersistentForms[1] : kPersistentForms[0];
}

} // namespace

cudaError_t ln_persistent_static_smem(int *bytes)
{
    cudaFuncAttributes a;
    // the forms declare the same static shared memory; report the largest
    int most = 0;
    for (const void *k : kPersistentForms) {
        const cudaError_t e = cudaFuncGetAttributes(&a, k);
        if (e != cudaSuccess)
            return e;
        most = static_cast<int>(a.sharedSizeBytes) > most ? static_cast<int>(a.sharedSizeBytes) : most;
    }
    *bytes = most;
    return cudaSuccess;
}

cudaError_t ln_persistent_setup(int max_dynamic_smem)
{
    for (const void *k : kPersistentForms) {
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dynamic_smem);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t ln_persistent_occupancy(int dyn_smem, int *ctas_per_sm)
{
    // the smallest over the forms (each is one CTA a SM by design)
    int least = 1 << 30;
    for (const void *k : kPersistentForms) {
        int n = 0;
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, LN_THREADS, dyn_smem);
        if (e != cudaSuccess)
            return e;
        least = n < least ? n : least;
    }
    *ctas_per_sm = least;
    return cudaSuccess;
}

cudaError_t ln_persistent_launch(const LnParams &p, int grid, int dyn_smem, cudaStream_t stream, bool bf16,
                                 const GnPersist *gn)
{
    LnParams args = p;
    GnPersist gargs = gn ? *gn : GnPersist{1, 1, 8, 0.f};
    void *kargs[] = {&args, &gargs};
    return cudaLaunchCooperativeKernel(persistent_form(bf16, gn != nullptr, p.groups == 1), dim3(grid),
                                       dim3(LN_THREADS), kargs, static_cast<size_t>(dyn_smem), stream);
}

int64_t ln_rows_max_row_len()
{
    return int64_t(512) * 8 * 4;
}

template <typename T, int NT>
cudaError_t ln_rows_launch_t(const LnParams &p, int sm_count, cudaStream_t stream)
{
    const int64_t L4 = p.row_len / 4;
    int64_t grid = p.rows;
    // Grid: up to 8192 / NT CTAs per SM in fp32 and 4096 / NT in bf16, i.e.
    // several waves of the resident CTAs (a CTA's rows run load -> reduce ->
    // store in turn, and CTAs that start as others finish overlap those
    // phases).  Measured back to back against 2048 / NT: fp32 (16384, 4096)
    // 85.8 -> 81.2 us, (65536, 1024) 86.2 -> 81.1 us; bf16 (16384, 4096)
    // 50.2 -> 47.7 us.  Larger grids lost on short rows (bf16 (65536, 1024)
    // 69.0 us at 16384 / NT).
    constexpr int64_t per_sm_threads = sizeof(T) == 2 ? 4096 : 8192;
    const int64_t cap = static_cast<int64_t>(sm_count) * (per_sm_threads / NT);
    if (grid > cap)
        grid = cap;
    const dim3 g(static_cast<unsigned>(grid));
    if (L4 <= NT)
        return launch_pdl(ln_rows_kernel<T, NT, 1>, g, dim3(NT), 0, stream, p);
    if (L4 <= 2 * NT)
        return launch_pdl(ln_rows_kernel<T, NT, 2>, g, dim3(NT), 0, stream, p);
    if (L4 <= 4 * NT)
        return launch_pdl(ln_rows_kernel<T, NT, 4>, g, dim3(NT), 0, stream, p);
    if (L4 <= 8 * NT)
        return launch_pdl(ln_rows_kernel<T, NT, 8>, g, dim3(NT), 0, stream, p);
    if (L4 <= 16 * NT)
        return launch_pdl(ln_rows_kernel<T, NT, 16>, g, dim3(NT), 0, stream, p);
    return cudaErrorInvalidValue;
}

// CTA size for a row of L4 vectors: the smallest of 32..512 threads that
// holds it with 8 vectors a thread, gamma/beta through L1.  Small CTAs keep many rows in flight per SM: the row lives in
// registers, so rows in flight are what hides the loads' latency.
template <typename T>
cudaError_t ln_rows_launch_sized(const LnParams &p, int sm_count, cudaStream_t stream)
{
    // vectors a thread: 8, or 16 for bf16 rows of more than 2,048 values
    // (held packed, so the same registers; 64 threads or more a row)
    const int64_t L4 = p.row_len / 4;
    const int64_t VT = sizeof(T) == 2 && L4 > 64 * 8 ? 16 : 8;
    if (L4 <= 32 * VT)
        return ln_rows_launch_t<T, 32>(p, sm_count, stream);
    if (L4 <= 64 * VT)
        return ln_rows_launch_t<T, 64>(p, sm_count, stream);
    if (L4 <= 128 * VT)
        return ln_rows_launch_t<T, 128>(p, sm_count, stream);
    if (L4 <= 256 * VT)
        return ln_rows_launch_t<T, 256>(p, sm_count, stream);
    return ln_rows_launch_t<T, 512>(p, sm_count, stream);
}

cudaError_t ln_rows_launch(const LnParams &p, bool bf16, int sm_count, cudaStream_t stream)
{
    return bf16 ? ln_rows_launch_sized<__nv_bfloat16>(p, sm_count, stream)
                : ln_rows_launch_sized<float>(p, sm_count, stream);
}

template <typename T>
cudaError_t ln_split_launch_t(const LnParams &p, bool vec4, cudaStream_t stream)
{
    dim3 grid(static_cast<unsigned>(p.parts), static_cast<unsigned>(p.rows < 65535 ? p.rows : 65535));
    cudaError_t e;
    if (vec4) {
        e = launch_pdl(ln_split_stats_kernel<T, true>, grid, dim3(LS_T), 0, stream, p);
        if (e == cudaSuccess)
            e = launch_pdl(ln_split_apply_kernel<T, true>, grid, dim3(LS_T), 0, stream, p);
    } else {
        e = launch_pdl(ln_split_stats_kernel<T, false>, grid, dim3(LS_T), 0, stream, p);
        if (e == cudaSuccess)
            e = launch_pdl(ln_split_apply_kernel<T, false>, grid, dim3(LS_T), 0, stream, p);
    }
    return e;
}

cudaError_t ln_split_launch(const LnParams &p, bool bf16, bool vec4, cudaStream_t stream)
{
    return bf16 ? ln_split_launch_t<__nv_bfloat16>(p, vec4, stream) : ln_split_launch_t<float>(p, vec4, stream);
}

cudaError_t ln_split_stats_launch(const LnParams &p, bool bf16, bool vec4, cudaStream_t stream)
{
    dim3 grid(static_cast<unsigned>(p.parts), static_cast<unsigned>(p.rows < 65535 ? p.rows : 65535));
    if (bf16)
        return vec4 ? launch_pdl(ln_split_stats_kernel<__nv_bfloat16, true>, grid, dim3(LS_T), 0, stream, p)
                    : launch_pdl(ln_split_stats_kernel<__nv_bfloat16, false>, grid, dim3(LS_T), 0, stream, p);
    return vec4 ? launch_pdl(ln_split_stats_kernel<float, true>, grid, dim3(LS_T), 0, stream, p)
                : launch_pdl(ln_split_stats_kernel<float, false>, grid, dim3(LS_T), 0, stream, p);
}

} // namespace normk
