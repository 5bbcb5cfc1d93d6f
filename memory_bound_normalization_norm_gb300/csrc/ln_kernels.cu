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
// co-resident).  CTA c owns the same float4 column slice of every row.  Row
// slices arrive by bulk copy (TMA engine, 32 KB pieces) into two
// shared-memory buffers, two rows ahead; the slice of the row being written
// lives in registers, and gamma/beta of the slice live in tensor memory
// (TMEM), loaded once per launch.  x is read from HBM once and stays on chip
// until y is written; gamma and beta are read from HBM once.  Warp 0
// coordinates the grid barrier; warps 1..15 own the data (warp 1 also issues
// the bulk copies).  Iteration r:
//   1. warps 1..15 reduce the triples of row r+1 from its buffer; barrier 1
//      (block-wide) also checks that warp 0 has merged row r;
//   2. warp 0 publishes the CTA's triple of row r+1, then, without waiting
//      for the data warps again, polls and merges row r+1 until the next
//      barrier 1, so the grid-wide exchange has a whole iteration to finish;
//   3. warps 1..15 write y of row r from registers and TMEM, move row r+1
//      from its buffer into registers, and warp 1 refills the buffer with
//      the bulk copy of row r+3.
// The pivot's three candidate elements travel with each row's bulk copy.
//
// Grid barrier without atomics.  Each CTA publishes its (mean, M2) as two
// 64-bit words, each carrying a 32-bit tag in its high half.  Both the
// record and the polls go through the bulk-copy unit (a 16-byte bulk store;
// one bulk load of all G records per attempt): plain loads and stores would
// queue behind the SM's own y stores, which drain at HBM speed.  The barrier
// and its data arrive in the same round trip.  Records sit in 4 rotating
// slots.  Tags count rows: row r of a launch is tagged row_base + r + 1,
// where row_base (workspace header) is the number of rows the persistent
// kernel has already processed on this workspace.  A slot therefore only
// ever holds tags smaller than the one awaited, and a zeroed workspace holds
// tag 0, which is never awaited.  row_base is read at kernel start and
// advanced by CTA 0 after its last merge, which proves every CTA has read
// it.  Every wait is bounded by %globaltimer: on timeout a CTA records
// NORM_ERR_TIMEOUT, drains its own bulk copies, frees its TMEM and returns
// without writing the remaining rows of y.
//
// Split path (any shape): kernel 1 writes one triple per (row, chunk) CTA;
// kernel 2 merges the row's triples and applies, re-reading x.
#include "norm_internal.cuh"

namespace normk {

namespace {

// Warp 0 coordinates; warps 1..15 own the row slice (15 float4 each).
constexpr int LN_DATA_WARPS = 15;
constexpr int LN_T = 32 * LN_DATA_WARPS;  // data threads
constexpr int LN_THREADS = LN_T + 32;     // CTA size
constexpr int LN_V = 15;                  // float4 of the slice per data thread
constexpr int LN_GB = 3;                  // gamma/beta float4 per TMEM load batch
constexpr int LN_NB = LN_V / LN_GB;       // batches per row
constexpr uint32_t LN_TMEM_COLS = 512;    // TMEM columns the CTA allocates (all)
constexpr int LN_TM_COLS = 8 * LN_V;      // TMEM columns of one data thread: gamma, beta
constexpr uint32_t LN_TM_BETA = 4 * LN_V; // column offset of beta within them
constexpr int LN_SLOTS = 4;               // partial-record slots: reused 4 rows later
constexpr int LN_MAX_GRID = 160;          // CTAs whose records one warp loads at once
constexpr uint32_t LN_BULK_CHUNK = 32768;
static_assert(LN_V % LN_GB == 0, "whole gamma/beta batches");
// warps 1..15 sit in TMEM quarters by warp % 4 and take column ranges by
// warp / 4, so at most four of them share a quarter
static_assert(4 * LN_TM_COLS <= static_cast<int>(LN_TMEM_COLS), "gamma/beta of a quarter fit TMEM");
static_assert(LN_DATA_WARPS + 1 <= 16, "warp / 4 < 4");

struct RowMean {
    float hi, lo, rstd;
};

// Fold `cnt` partials part[0..cnt) = (n, mean of x - K_i, M2, K_i) in a
// fixed order with one warp; every mean is first re-expressed against K_ref.
// All lanes return the same result.  Count-weighted, so empty partials are
// harmless.
__device__ __forceinline__ Moments merge_partials_warp(const float4 *part, int cnt, float K_ref)
{
    const int lane = threadIdx.x & 31;
    Moments acc = {0.f, 0.f, 0.f};
    for (int i = lane; i < cnt; i += 32) {
        const float4 q = ld_l2_f4(part + i);
        const Moments m = {q.x, (q.w - K_ref) + q.y, q.z};
        chan_merge(acc, m);
    }
    return warp_merge(acc);
}

__device__ __forceinline__ RowMean finish_row(float K, const Moments &tot, float eps)
{
    // mean = K + tot.mean, kept as an exact two-term sum (Knuth TwoSum).
    const float s = K + tot.mean;
    const float bp = s - K;
    const float err = (K - (s - bp)) + (tot.mean - bp);
    const float var = fmaxf(tot.m2 / tot.n, 0.f);
    RowMean rm;
    rm.hi = s;
    rm.lo = err;
    rm.rstd = rsqrtf(var + eps);
    return rm;
}

__device__ __forceinline__ float4 ln_apply4(float4 v, const RowMean &rm, float4 g, float4 b)
{
    float4 o;
    o.x = fmaf(((v.x - rm.hi) - rm.lo) * rm.rstd, g.x, b.x);
    o.y = fmaf(((v.y - rm.hi) - rm.lo) * rm.rstd, g.y, b.y);
    o.z = fmaf(((v.z - rm.hi) - rm.lo) * rm.rstd, g.z, b.z);
    o.w = fmaf(((v.w - rm.hi) - rm.lo) * rm.rstd, g.w, b.w);
    return o;
}

// CTA-wide fold of per-thread triples; the result is valid in thread 0.
template <int T>
__device__ __forceinline__ Moments cta_merge(Moments m, Moments *scratch)
{
    m = warp_merge(m);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        scratch[warp] = m;
    __syncthreads();
    Moments r = {0.f, 0.f, 0.f};
    if (warp == 0) {
        if (lane < T / 32)
            r = scratch[lane];
        r = warp_merge(r);
    }
    return r;
}

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
// with each count n_c known from the partition (q4 or q4 + 1 float4).  The
// sums are warp reductions in a fixed order, so every CTA computes the same
// bits; all lanes return the result.
__device__ __forceinline__ Moments merge_records(const unsigned long long (&w)[LN_MAX_GRID / 32][2], int G,
                                                 unsigned q4, unsigned rem)
{
    constexpr int J = LN_MAX_GRID / 32;
    const int lane = threadIdx.x & 31;
    const float N = 4.f * (static_cast<float>(q4) * static_cast<float>(G) + static_cast<float>(rem));
    float sm = 0.f; // sum of n_c * m_c
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int i = lane + 32 * j;
        if (i < G) {
            const float n = 4.f * static_cast<float>(q4 + (static_cast<unsigned>(i) < rem ? 1u : 0u));
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
            const float n = 4.f * static_cast<float>(q4 + (static_cast<unsigned>(i) < rem ? 1u : 0u));
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

// Warp 0: read the G records of a row until every tag equals `tag`
// (bounded by timeout_ns), then merge them.
//
// BULK = false: plain L2 loads (ld.global.cg), which overlap.  BULK = true:
// one bulk copy (TMA unit) of all records into rec_s per attempt, completed
// on `bar`; `phase` is the parity of bar's next completion and `inflight`
// tells the caller that a copy into rec_s may still be running after a
// timeout, which it must drain before exit.
template <bool BULK>
__device__ __forceinline__ GridMerge poll_and_merge(const unsigned long long *rec, unsigned long long *rec_s,
                                                    uint64_t *bar, uint32_t &phase, bool &inflight, int G,
                                                    unsigned q4, unsigned rem, unsigned tag, uint64_t timeout_ns,
                                                    uint64_t pol)
{
    constexpr int J = LN_MAX_GRID / 32;
    const int lane = threadIdx.x & 31;
    GridMerge g;
    g.ok = true;
    uint64_t t0 = 0;
    for (int attempt = 0;; ++attempt) {
        if (BULK) {
            int landed = 0;
            if (lane == 0) {
                // the warp's reads of the previous attempt precede the copy
                fence_proxy_async_smem();
                const uint32_t bytes = static_cast<uint32_t>(G) * 16u;
                mbar_arrive_expect_tx(bar, bytes);
                bulk_g2s(rec_s, rec, bytes, bar, pol);
                inflight = true;
                landed = mbar_wait_bounded(bar, phase, timeout_ns) ? 1 : 0;
                if (landed) {
                    inflight = false;
                    phase ^= 1u;
                }
            }
            if (!__shfl_sync(0xffffffffu, landed, 0)) {
                g.ok = false;
                return g;
            }
            __syncwarp();
        }
        // the words live only inside one attempt, so they stay in registers
        unsigned long long w[J][2];
        unsigned bad = 0;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            // lanes past the last CTA re-read record G-1 (branch-free loads)
            const int i = min(lane + 32 * j, G - 1);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                w[j][e] = BULK ? rec_s[2 * i + e] : ld_cg_u64(rec + 2 * i + e);
                bad |= record_tag(w[j][e]) ^ tag;
            }
        }
        if (__all_sync(0xffffffffu, bad == 0)) {
            g.tot = merge_records(w, G, q4, rem);
            return g;
        }
        if (attempt == 0)
            t0 = globaltimer_ns();
        else if (__any_sync(0xffffffffu, globaltimer_ns() - t0 > timeout_ns)) {
            g.ok = false;
            return g;
        }
        if (BULK)
            __syncwarp();
        else
            __nanosleep(20);
    }
}

// Pivot of a row: the median of its first, middle and last elements.  A
// pivot inside the bulk of the row keeps the shifted sums small, and one
// outlier cannot become the pivot.  The three elements arrive by bulk copy
// with the row, each in the 16-byte piece that contains it (row_len is a
// multiple of 4, so element i sits at float i % 4 of piece i / 4).
__device__ __forceinline__ float row_pivot(const float4 *piece, int64_t row_len)
{
    const int64_t mid = row_len >> 1;
    const float a = piece[0].x;
    const float4 pm = piece[1], pl = piece[2];
    const int jm = static_cast<int>(mid & 3);
    const float b = jm == 0 ? pm.x : jm == 1 ? pm.y : jm == 2 ? pm.z : pm.w;
    const float c = pl.w; // row_len - 1 is float 3 of its piece
    return fmaxf(fminf(a, b), fminf(fmaxf(a, b), c));
}

#ifndef LN_BULK_BARRIER
#define LN_BULK_BARRIER 1
#endif
// How the grid barrier's records travel: plain loads and stores (0) or bulk
// copies (1).
constexpr bool LN_BULK_RECORDS = LN_BULK_BARRIER != 0;

// Named barriers of the persistent kernel (0 is __syncthreads).
constexpr int LN_BAR_PUBLISHED = 1; // warp 0 has issued the row's record
constexpr int LN_BAR_ROW_DONE = 2;  // y of row r written, row r+1 in registers

__global__ void __launch_bounds__(LN_THREADS, 1) ln_persistent_kernel(LnParams p)
{
    extern __shared__ __align__(128) float4 ln_smem[];
    __shared__ __align__(8) uint64_t bar_x[2];
    __shared__ Moments red[LN_DATA_WARPS];
    __shared__ float4 piv_in[2][3]; // pieces holding a row's pivot candidates, by row parity
    __shared__ RowMean row_mean[2]; // merged statistics of a row, by row parity
    __shared__ unsigned row_base_s;
    __shared__ uint32_t tmem_base_s;
    __shared__ __align__(8) uint64_t bar_rec;                             // record fetches (bulk)
    __shared__ __align__(16) unsigned long long rec_in[LN_BULK_RECORDS ? 2 * LN_MAX_GRID : 2];
    __shared__ __align__(16) unsigned long long rec_out[2];               // this CTA's record (bulk)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int64_t R = p.rows;
    const int64_t L4 = p.row_len >> 2;
    // CTA c owns n4 = q4 (+1 for the first rem CTAs) float4 of every row,
    // starting at f0; the merge recomputes every CTA's count the same way.
    const unsigned q4 = static_cast<unsigned>(L4 / G), rem = static_cast<unsigned>(L4 % G);
    const int64_t f0 = static_cast<int64_t>(cta) * q4 + min(static_cast<unsigned>(cta), rem);
    const int n4 = static_cast<int>(q4 + (static_cast<unsigned>(cta) < rem ? 1u : 0u));
    const float4 *x4 = reinterpret_cast<const float4 *>(p.x);
    float4 *y4 = reinterpret_cast<float4 *>(p.y);
    const float4 *g4 = reinterpret_cast<const float4 *>(p.gamma);
    const float4 *b4 = reinterpret_cast<const float4 *>(p.beta);
    unsigned long long *records = reinterpret_cast<unsigned long long *>(p.part);
    const int buf_f4 = (p.max_n4 + 7) & ~7;

    const uint64_t pol_stream = policy_evict_first();

    // The CTA holds all 512 TMEM columns (it is alone on its SM: its 512
    // threads at 128 registers take the whole register file).
    if (warp == 0)
        tmem_alloc(&tmem_base_s, LN_TMEM_COLS);
    if (tid == 0) {
        mbar_init(&bar_x[0], 1);
        mbar_init(&bar_x[1], 1);
        mbar_init(&bar_rec, 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        row_base_s = ld_relaxed_gpu_u32(&p.sync->row_base);
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const unsigned row_base = row_base_s;
    const uint32_t tmem_base = tmem_base_s;
    bool aborted = false;

    // Warp 0 and warps 1..15 run separate loops.  Per iteration r both pass
    // the block-wide barrier 1 (__syncthreads_or: abort vote; the triples of
    // row r+1 are reduced and row r is merged) and the named barriers
    // LN_BAR_PUBLISHED and LN_BAR_ROW_DONE, at which warp 0 only arrives: it
    // goes on merging row r+1 until the next barrier 1.
    if (warp == 0) {
        // ------------------------------------------------ coordinator
        uint32_t rec_phase = 0;    // parity of bar_rec's next completion
        bool rec_inflight = false; // a record fetch may still be writing rec_in
        const uint64_t pol_rec = policy_evict_last();
        bool fail = false;         // the merge of the previous row gave up
        for (int64_t r = -1; r < R; ++r) {
            const int64_t nx = r + 1;
            if (__syncthreads_or(fail ? 1 : 0)) { // 1
                aborted = true;
                break;
            }
            if (nx < R) {
                Moments c = {0.f, 0.f, 0.f};
                if (lane < LN_DATA_WARPS)
                    c = red[lane];
                c = warp_merge(c);
                // read now: the bulk copy of row nx + 2, issued after
                // LN_BAR_ROW_DONE, overwrites these pieces.  (The data warps
                // saw row nx land before barrier 1; this wait returns at once
                // and orders the read after the copy for this warp as well.)
                fail = !mbar_wait_bounded(&bar_x[nx & 1], static_cast<uint32_t>((nx >> 1) & 1), p.timeout_ns);
                const float K = row_pivot(piv_in[nx & 1], p.row_len);
                const unsigned tag = row_tag(row_base, nx);
                unsigned long long *slot = records + static_cast<int64_t>(nx % LN_SLOTS) * G * 2;
                if (lane == 0) {
                    if (LN_BULK_RECORDS) {
                        bulk_wait_read_all(); // the previous record has left rec_out
                        rec_out[0] = tagged(tag, c.mean);
                        rec_out[1] = tagged(tag, c.m2);
                        fence_proxy_async_smem();
                        bulk_s2g(slot + 2 * cta, rec_out, 16);
                        bulk_commit();
                    } else {
                        st_relaxed_gpu_u64(slot + 2 * cta + 0, tagged(tag, c.mean));
                        st_relaxed_gpu_u64(slot + 2 * cta + 1, tagged(tag, c.m2));
                    }
                }
                __syncwarp();
                bar_arrive_named(LN_BAR_PUBLISHED, LN_THREADS);
                bar_arrive_named(LN_BAR_ROW_DONE, LN_THREADS);
                // merge row nx while the data warps write row r and reduce
                // row nx + 1; due at the next barrier 1
                const GridMerge gm = poll_and_merge<LN_BULK_RECORDS>(slot, rec_in, &bar_rec, rec_phase, rec_inflight,
                                                                     G, q4, rem, tag + p.tag_skew, p.timeout_ns,
                                                                     pol_rec);
                if (!gm.ok || fail) {
                    fail = true;
                    if (lane == 0)
                        record_error(p.err, NORM_ERR_TIMEOUT);
                } else if (lane == 0) {
                    row_mean[nx & 1] = finish_row(K, gm.tot, p.eps);
                    // every CTA has read row_base once CTA 0 has merged the last row
                    if (nx + 1 == R && cta == 0)
                        st_relaxed_gpu_u32(&p.sync->row_base, row_base + static_cast<unsigned>(R));
                }
            } else {
                bar_arrive_named(LN_BAR_PUBLISHED, LN_THREADS);
                bar_arrive_named(LN_BAR_ROW_DONE, LN_THREADS);
            }
        }
        if (lane == 0) {
            // never leave a bulk copy in flight into or out of shared memory
            if (rec_inflight && !mbar_wait_bounded(&bar_rec, rec_phase, p.timeout_ns))
                record_error(p.err, NORM_ERR_TIMEOUT);
            if (LN_BULK_RECORDS)
                bulk_wait_all();
            if (aborted)
                record_error(p.err, NORM_ERR_TIMEOUT);
        }
    } else {
        // ------------------------------------------------ data warps 1..15
        const int dt = tid - 32;
        // Thread 32 (warp 1, lane 0) issues the bulk copies of x.  It tracks
        // those it issued (rows < issued) and those whose completion it
        // observed (rows < waited), so that an early exit can drain them.
        const bool issuer = dt == 0;
        int64_t issued = 0, waited = 0;
        // Row q's slice, plus the three 16-byte pieces of the row that hold
        // its pivot candidates, all on bar_x[q & 1].
        auto issue_x = [&](int64_t q) {
            uint64_t *bar = &bar_x[q & 1];
            const uint32_t bytes = static_cast<uint32_t>(n4) * 16u;
            mbar_arrive_expect_tx(bar, bytes + 48u);
            const float4 *row = x4 + q * L4;
            bulk_g2s(&piv_in[q & 1][0], row, 16u, bar, pol_stream);
            bulk_g2s(&piv_in[q & 1][1], row + ((p.row_len >> 1) >> 2), 16u, bar, pol_stream);
            bulk_g2s(&piv_in[q & 1][2], row + (L4 - 1), 16u, bar, pol_stream);
            const float4 *src = row + f0;
            float4 *dst = ln_smem + (q & 1) * buf_f4;
            for (uint32_t off = 0; off < bytes; off += LN_BULK_CHUNK)
                bulk_g2s(dst + off / 16, src + off / 16,
                         (bytes - off < LN_BULK_CHUNK) ? (bytes - off) : LN_BULK_CHUNK, bar, pol_stream);
            issued = q + 1;
        };
        if (issuer) {
            issue_x(0);
            if (R > 1)
                issue_x(1);
        }
        // This thread's TMEM cells: lane 32*(warp % 4) + lane of its warp's
        // quarter, LN_TM_COLS columns from (warp / 4) * LN_TM_COLS: gamma of
        // its k-th float4 at column 4k, beta at LN_TM_BETA + 4k.  The four
        // (or three) data warps of a quarter take disjoint column ranges.
        const uint32_t tm = tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16) +
                            static_cast<uint32_t>((warp >> 2) * LN_TM_COLS);
        float4 v[LN_V]; // this thread's part of the slice of row r
        for (int64_t r = -1; r < R; ++r) {
            const int64_t nx = r + 1;

            // 1. triple of row nx from its shared-memory buffer, about the
            //    row's pivot K
            bool fail = false;
            if (nx < R) {
                const float4 *buf = ln_smem + (nx & 1) * buf_f4;
                if (!mbar_wait_bounded(&bar_x[nx & 1], static_cast<uint32_t>((nx >> 1) & 1), p.timeout_ns)) {
                    fail = true;
                } else {
                    if (issuer)
                        waited = nx + 1;
                    const float K = row_pivot(piv_in[nx & 1], p.row_len);
                    // one pass over shared memory: shifted sums of d = x - K
                    float s1 = 0.f, s2 = 0.f;
                    int cnt = 0;
#pragma unroll
                    for (int k = 0; k < LN_V; ++k) {
                        const int i = dt + k * LN_T;
                        if (i < n4) {
                            const float4 q = buf[i];
                            const float a = q.x - K, bq = q.y - K, c = q.z - K, d = q.w - K;
                            s1 += (a + bq) + (c + d);
                            s2 = fmaf(a, a, fmaf(bq, bq, fmaf(c, c, fmaf(d, d, s2))));
                            cnt += 4;
                        }
                    }
                    Moments m = {0.f, 0.f, 0.f};
                    if (cnt > 0) {
                        m.n = static_cast<float>(cnt);
                        m.mean = s1 / m.n;
                        m.m2 = fmaxf(fmaf(-s1, m.mean, s2), 0.f);
                    }
                    m = warp_merge(m);
                    if (lane == 0)
                        red[warp - 1] = m;
                }
            }
            if (__syncthreads_or(fail ? 1 : 0)) { // 1
                aborted = true;
                break;
            }
            // the CTA's record of row nx goes out before this CTA's y stores
            bar_sync_named(LN_BAR_PUBLISHED, LN_THREADS);

            if (r < 0) {
                // 2'. before the first row: gamma and beta of the slice go to
                //     TMEM once, staged through v (free until row 0 arrives)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float4 *src = h == 0 ? g4 : b4;
                    const float4 dflt = h == 0 ? make_float4(1.f, 1.f, 1.f, 1.f) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < LN_V; ++k) {
                        const int i = dt + k * LN_T;
                        v[k] = (src && i < n4) ? ld_stream_f4(src + f0 + i, pol_stream) : dflt;
                    }
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < LN_V; ++k)
                        tmem_st4(tm + static_cast<uint32_t>(h * LN_TM_BETA + 4 * k), v[k]);
                    tmem_wait_st();
                }
            } else {
                // 2. y of row r from registers, gamma/beta from TMEM, one
                //    batch of LN_GB float4 loaded while the previous one is
                //    written
                const RowMean rm = row_mean[r & 1];
                float4 *yr = y4 + r * L4 + f0;
                float4 gA[LN_GB], bA[LN_GB], gB[LN_GB], bB[LN_GB];
                // tcgen05 loads and waits are warp-collective: reconverge
                // after the divergent stores first
                auto load_gb = [&](int bt, float4 *g, float4 *bb) {
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < LN_GB; ++j) {
                        const uint32_t c = static_cast<uint32_t>(4 * (bt * LN_GB + j));
                        g[j] = tmem_ld4(tm + c);
                        bb[j] = tmem_ld4(tm + LN_TM_BETA + c);
                    }
                };
                auto pin_gb = [&](float4 *g, float4 *bb) {
                    __syncwarp();
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < LN_GB; ++j) {
                        tmem_pin(g[j]);
                        tmem_pin(bb[j]);
                    }
                };
                auto write_batch = [&](int bt, const float4 *g, const float4 *bb) {
#pragma unroll
                    for (int j = 0; j < LN_GB; ++j) {
                        const int k = bt * LN_GB + j;
                        const int i = dt + k * LN_T;
                        if (i < n4)
                            st_stream_f4(yr + i, ln_apply4(v[k], rm, g[j], bb[j]), pol_stream);
                    }
                };
                load_gb(0, gA, bA);
                pin_gb(gA, bA);
                // batches alternate between the A and B registers (the branch on
                // bt's parity is resolved at compile time)
#pragma unroll
                for (int bt = 0; bt < LN_NB; ++bt) {
                    if ((bt & 1) == 0) {
                        if (bt + 1 < LN_NB)
                            load_gb(bt + 1, gB, bB);
                        write_batch(bt, gA, bA);
                        if (bt + 1 < LN_NB)
                            pin_gb(gB, bB);
                    } else {
                        if (bt + 1 < LN_NB)
                            load_gb(bt + 1, gA, bA);
                        write_batch(bt, gB, bB);
                        if (bt + 1 < LN_NB)
                            pin_gb(gA, bA);
                    }
                }
            }
            // row nx moves into registers
            if (nx < R) {
                const float4 *buf = ln_smem + (nx & 1) * buf_f4;
#pragma unroll
                for (int k = 0; k < LN_V; ++k) {
                    const int i = dt + k * LN_T;
                    v[k] = (i < n4) ? buf[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            __syncwarp();
            bar_sync_named(LN_BAR_ROW_DONE, LN_THREADS);
            // buffer nx & 1 and its pivot pieces are free: refill them
            if (issuer && nx + 2 < R) {
                fence_proxy_async_smem();
                issue_x(nx + 2);
            }
        }
        // Drain: never leave a bulk copy in flight into shared memory.
        if (issuer) {
            for (int64_t q = waited; q < issued; ++q) {
                if (!mbar_wait_bounded(&bar_x[q & 1], static_cast<uint32_t>((q >> 1) & 1), p.timeout_ns))
                    record_error(p.err, NORM_ERR_TIMEOUT);
            }
        }
    }
    // Every TMEM access of every thread is complete before warp 0 frees it.
    tmem_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tmem_fence_after_sync();
        tmem_dealloc(tmem_base, LN_TMEM_COLS);
    }
}

// ---------------------------------------------------------------- split path

constexpr int LS_T = 256;

// One triple per (chunk p, row r) CTA.  Vector form folds each float4 as a
// two-pass group of 4 into the thread's triple; scalar form is Welford.
template <bool VEC>
__global__ void __launch_bounds__(LS_T) ln_split_stats_kernel(LnParams p)
{
    __shared__ Moments red[LS_T / 32];
    const int P = p.parts;
    for (int64_t r = blockIdx.y; r < p.rows; r += gridDim.y) {
        const int pc = blockIdx.x;
        const float *xr = p.x + r * p.row_len;
        const float K = ld_plain_f1(xr);
        const int64_t lo = static_cast<int64_t>(pc) * p.chunk;
        const int64_t hi = (lo + p.chunk < p.row_len) ? lo + p.chunk : p.row_len;
        Moments m = {0.f, 0.f, 0.f};
        if (VEC) {
            const uint64_t pol = policy_evict_first();
            const float4 *x4 = reinterpret_cast<const float4 *>(xr);
            for (int64_t i = lo / 4 + threadIdx.x; i < hi / 4; i += LS_T) {
                const float4 q = ld_stream_f4(x4 + i, pol);
                const float a = q.x - K, b = q.y - K, c = q.z - K, d = q.w - K;
                Moments g;
                g.n = 4.f;
                g.mean = ((a + b) + (c + d)) * 0.25f;
                const float da = a - g.mean, db = b - g.mean, dc = c - g.mean, dd = d - g.mean;
                g.m2 = (da * da + db * db) + (dc * dc + dd * dd);
                chan_merge(m, g);
            }
        } else {
            for (int64_t i = lo + threadIdx.x; i < hi; i += LS_T) {
                const float d = ld_plain_f1(xr + i) - K;
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

template <bool VEC>
__global__ void __launch_bounds__(LS_T) ln_split_apply_kernel(LnParams p)
{
    __shared__ RowMean row_mean;
    const int P = p.parts;
    for (int64_t r = blockIdx.y; r < p.rows; r += gridDim.y) {
        const int pc = blockIdx.x;
        const float *xr = p.x + r * p.row_len;
        float *yr = p.y + r * p.row_len;
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
            const float4 *x4 = reinterpret_cast<const float4 *>(xr);
            float4 *y4 = reinterpret_cast<float4 *>(yr);
            const float4 *g4 = reinterpret_cast<const float4 *>(p.gamma);
            const float4 *b4 = reinterpret_cast<const float4 *>(p.beta);
            for (int64_t i = lo / 4 + threadIdx.x; i < hi / 4; i += LS_T) {
                const float4 q = ld_stream_f4(x4 + i, pol);
                const float4 g = g4 ? ld_ro_f4(g4 + i, pol_gb) : make_float4(1.f, 1.f, 1.f, 1.f);
                const float4 bb = b4 ? ld_ro_f4(b4 + i, pol_gb) : make_float4(0.f, 0.f, 0.f, 0.f);
                st_stream_f4(y4 + i, ln_apply4(q, rm, g, bb), pol);
            }
        } else {
            for (int64_t i = lo + threadIdx.x; i < hi; i += LS_T) {
                const float g = p.gamma ? p.gamma[i] : 1.f;
                const float bb = p.beta ? p.beta[i] : 0.f;
                yr[i] = fmaf(((ld_plain_f1(xr + i) - rm.hi) - rm.lo) * rm.rstd, g, bb);
            }
        }
        __syncthreads();
    }
}

} // namespace

LnPersistentConfig ln_persistent_config()
{
    return LnPersistentConfig{LN_THREADS, LN_T, LN_V, LN_SLOTS * 16, LN_MAX_GRID};
}

cudaError_t ln_persistent_static_smem(int *bytes)
{
    cudaFuncAttributes a;
    const cudaError_t e = cudaFuncGetAttributes(&a, ln_persistent_kernel);
    if (e == cudaSuccess)
        *bytes = static_cast<int>(a.sharedSizeBytes);
    return e;
}

cudaError_t ln_persistent_setup(int max_dynamic_smem)
{
    return cudaFuncSetAttribute(ln_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                max_dynamic_smem);
}

cudaError_t ln_persistent_occupancy(int dyn_smem, int *ctas_per_sm)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, ln_persistent_kernel, LN_THREADS, dyn_smem);
}

cudaError_t ln_persistent_launch(const LnParams &p, int grid, int dyn_smem, cudaStream_t stream)
{
    LnParams args = p;
    void *kargs[] = {&args};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(ln_persistent_kernel), dim3(grid),
                                       dim3(LN_THREADS), kargs, static_cast<size_t>(dyn_smem), stream);
}

cudaError_t ln_split_launch(const LnParams &p, bool vec4, cudaStream_t stream)
{
    dim3 grid(static_cast<unsigned>(p.parts), static_cast<unsigned>(p.rows < 65535 ? p.rows : 65535));
    if (vec4) {
        ln_split_stats_kernel<true><<<grid, LS_T, 0, stream>>>(p);
        ln_split_apply_kernel<true><<<grid, LS_T, 0, stream>>>(p);
    } else {
        ln_split_stats_kernel<false><<<grid, LS_T, 0, stream>>>(p);
        ln_split_apply_kernel<false><<<grid, LS_T, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

} // namespace normk
