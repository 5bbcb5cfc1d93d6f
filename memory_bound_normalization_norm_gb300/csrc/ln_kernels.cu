// ln_kernels.cu - LayerNorm over long contiguous rows (LayerNorm page,
// POPCORNBENCH transcript "Kimi-K2.6 l1_p40": per row, mean and population
// variance over the normalized extent, y = (x - mean)/sqrt(var + eps) *
// gamma + beta with elementwise gamma/beta).
//
// Statistics.  All partial statistics are (count, mean, M2) triples of
// d = x - K, where the pivot K is an element of the row (the first element
// of the CTA's slice in the persistent kernel, x[r][0] in the split path).
// Shifting by an element of the row keeps the partial sums small when
// |mean| >> std (for x ~ N(1000, 0.01^2) an fp32 sum of raw x would lose the
// variance entirely); d is exact whenever x and K are within a factor of 2.
// Per thread the triple is computed two-pass from registers, then folded with
// Chan's pairwise update (Chan, Golub, LeVeque 1979) across the warp, the CTA
// and finally across all CTAs of the row in a fixed order, each CTA's mean
// first re-expressed against one reference pivot K_ref ((K_c - K_ref) is
// exact for clustered data).  The row mean is then K_ref + delta, carried as
// an unevaluated fp32 pair (hi, lo), and the output is
// ((x - hi) - lo) * rstd * gamma + beta.
//
// Persistent path (one CTA per SM, cooperative launch so all CTAs are
// co-resident).  CTA c owns the same float4 column slice of every row.  For
// row r it:
//   1. waits for its slice, bulk-copied (TMA engine) into shared-memory
//      buffer r%2, and moves it into registers (V float4 per thread);
//   2. immediately reuses the buffer for the bulk copy of row r+2, so two
//      future rows stream from HBM while row r is reduced and written;
//   3. reduces its triple and publishes it to the workspace, then waits at a
//      per-row grid barrier (acquire/release counters, bounded by
//      %globaltimer: on timeout it records NORM_ERR_TIMEOUT, drains its own
//      bulk copies and returns without writing y);
//   4. merges all CTAs' triples (identically in every CTA) and writes y from
//      the registers with evict-first stores; gamma/beta are read through L2
//      with an evict-last policy so they come from HBM once per launch.
// x is read from HBM once and y written once.
//
// Split path (any shape): kernel 1 writes one triple per (row, chunk) CTA;
// kernel 2 merges the row's triples and applies, re-reading x.
#include "norm_internal.cuh"

namespace normk {

namespace {

constexpr int LN_T = 512; // threads per CTA, persistent kernel
constexpr int LN_V = 14;  // float4 per thread held in registers
constexpr int LN_AB = 5;  // gamma/beta float4 loaded ahead per batch
constexpr uint32_t LN_BULK_CHUNK = 32768;

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

__global__ void __launch_bounds__(LN_T, 1) ln_persistent_kernel(LnParams p)
{
    extern __shared__ __align__(128) float4 ln_smem[];
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ Moments red[LN_T / 32];
    __shared__ RowMean row_mean;

    const int tid = threadIdx.x;
    const int G = gridDim.x, cta = blockIdx.x;
    const int64_t L4 = p.row_len >> 2;
    const int64_t f0 = (static_cast<int64_t>(cta) * L4) / G;
    const int64_t f1 = (static_cast<int64_t>(cta + 1) * L4) / G;
    const int n4 = static_cast<int>(f1 - f0);
    const float4 *x4 = reinterpret_cast<const float4 *>(p.x);
    float4 *y4 = reinterpret_cast<float4 *>(p.y);
    const float4 *g4 = reinterpret_cast<const float4 *>(p.gamma);
    const float4 *b4 = reinterpret_cast<const float4 *>(p.beta);

    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();

    // Thread 0 tracks the bulk copies it issued (rows < issued) and those
    // already consumed (rows < consumed) so that an early exit can drain them.
    // Abort decisions are block-wide votes (__syncthreads_or), so every thread
    // leaves the row loop at the same barrier.
    int64_t issued = 0, consumed = 0;
    bool aborted = false;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    auto issue_row = [&](int64_t r) {
        uint64_t *bar = &bars[r & 1];
        const uint32_t bytes = static_cast<uint32_t>(n4) * 16u;
        mbar_arrive_expect_tx(bar, bytes);
        const float4 *src = x4 + r * L4 + f0;
        float4 *dst = ln_smem + ((r & 1) ? p.max_n4 : 0);
        for (uint32_t off = 0; off < bytes; off += LN_BULK_CHUNK) {
            const uint32_t nb = (bytes - off < LN_BULK_CHUNK) ? (bytes - off) : LN_BULK_CHUNK;
            bulk_g2s(dst + off / 16, src + off / 16, nb, bar, pol_stream);
        }
    };

    if (tid == 0) {
        issue_row(0);
        issued = 1;
        if (p.rows > 1) {
            issue_row(1);
            issued = 2;
        }
    }

    for (int64_t r = 0; r < p.rows; ++r) {
        const int b = static_cast<int>(r & 1);
        const uint32_t parity = static_cast<uint32_t>((r >> 1) & 1);
        const bool last_row = (r + 1 == p.rows);

        // 1. slice of row r -> registers
        const bool landed = mbar_wait_bounded(&bars[b], parity, p.timeout_ns);
        const float4 *cur = ln_smem + (b ? p.max_n4 : 0);
        // this CTA's pivot: the first element of its slice (any element of
        // the row serves; a CTA without elements contributes nothing)
        const float K = (n4 > 0) ? cur[0].x : 0.f;
        float4 v[LN_V];
#pragma unroll
        for (int k = 0; k < LN_V; ++k) {
            const int i = tid + k * LN_T;
            v[k] = (i < n4) ? cur[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // everyone has read the buffer; leave together if any wait gave up
        if (__syncthreads_or(landed ? 0 : 1)) {
            aborted = true;
            break;
        }
        if (tid == 0) {
            consumed = r + 1;
            // 2. refill the buffer with row r+2 while row r is processed
            if (r + 2 < p.rows) {
                fence_proxy_async_smem();
                issue_row(r + 2);
                issued = r + 3;
            }
        }

        // 3. per-thread two-pass triple of d = x - K over valid elements
        Moments m = {0.f, 0.f, 0.f};
        {
            float s = 0.f;
            int cnt = 0;
#pragma unroll
            for (int k = 0; k < LN_V; ++k) {
                if (tid + k * LN_T < n4) {
                    s += ((v[k].x - K) + (v[k].y - K)) + ((v[k].z - K) + (v[k].w - K));
                    cnt += 4;
                }
            }
            if (cnt > 0) {
                m.n = static_cast<float>(cnt);
                m.mean = s / m.n;
                float q = 0.f;
#pragma unroll
                for (int k = 0; k < LN_V; ++k) {
                    if (tid + k * LN_T < n4) {
                        const float a = (v[k].x - K) - m.mean, bq = (v[k].y - K) - m.mean;
                        const float c = (v[k].z - K) - m.mean, d = (v[k].w - K) - m.mean;
                        q = fmaf(a, a, q);
                        q = fmaf(bq, bq, q);
                        q = fmaf(c, c, q);
                        q = fmaf(d, d, q);
                    }
                }
                m.m2 = q;
            }
        }
        const Moments cm = cta_merge<LN_T>(m, red);

        // publish + grid barrier (thread 0), then merge of all partials (warp 0)
        bool ok = true;
        if (tid < 32) {
            float4 *slot = p.part + static_cast<int64_t>(b) * G;
            if (tid == 0) {
                const unsigned gen0 = ld_acquire_gpu(&p.sync->gen[b]);
                slot[cta] = make_float4(cm.n, cm.mean, cm.m2, K);
                const unsigned old = atom_add_acq_rel_gpu(&p.sync->count[b], 1u);
                if (old + 1 == p.expected) {
                    st_relaxed_gpu(&p.sync->count[b], 0u);
                    red_add_release_gpu(&p.sync->gen[b], 1u);
                } else {
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_gpu(&p.sync->gen[b]) == gen0) {
                        if (globaltimer_ns() - t0 > p.timeout_ns) {
                            ok = false;
                            break;
                        }
                        __nanosleep(32);
                    }
                }
                if (!ok)
                    record_error(p.err, NORM_ERR_TIMEOUT);
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            __syncwarp();
            if (ok) {
                // reference pivot: the last CTA's (its slice is never empty)
                const float K_ref = ld_l2_f4(slot + (G - 1)).w;
                const Moments tot = merge_partials_warp(slot, G, K_ref);
                if (tid == 0)
                    row_mean = finish_row(K_ref, tot, p.eps);
            }
        }
        if (__syncthreads_or(ok ? 0 : 1)) {
            aborted = true;
            break;
        }

        // 4. apply from registers; gamma/beta are loaded LN_AB float4 at a
        //    time ahead of the stores that need them
        const RowMean rm = row_mean;
        const uint64_t pol_gb = last_row ? pol_stream : pol_keep;
        float4 *yr = y4 + r * L4 + f0;
#pragma unroll
        for (int k0 = 0; k0 < LN_V; k0 += LN_AB) {
            float4 g[LN_AB], bb[LN_AB];
#pragma unroll
            for (int j = 0; j < LN_AB; ++j) {
                const int i = tid + (k0 + j) * LN_T;
                const bool in = (k0 + j < LN_V) && i < n4;
                g[j] = (in && g4) ? ld_ro_f4(g4 + f0 + i, pol_gb) : make_float4(1.f, 1.f, 1.f, 1.f);
                bb[j] = (in && b4) ? ld_ro_f4(b4 + f0 + i, pol_gb) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < LN_AB; ++j) {
                const int i = tid + (k0 + j) * LN_T;
                if ((k0 + j < LN_V) && i < n4)
                    st_stream_f4(yr + i, ln_apply4(v[k0 + j], rm, g[j], bb[j]), pol_stream);
            }
        }
    }

    // Drain: never leave a bulk copy in flight into shared memory.
    if (tid == 0) {
        for (int64_t q = consumed; q < issued; ++q) {
            if (!mbar_wait_bounded(&bars[q & 1], static_cast<uint32_t>((q >> 1) & 1), p.timeout_ns))
                record_error(p.err, NORM_ERR_TIMEOUT);
        }
        if (aborted)
            record_error(p.err, NORM_ERR_TIMEOUT);
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
    return LnPersistentConfig{LN_T, LN_V};
}

cudaError_t ln_persistent_setup(int max_dynamic_smem)
{
    return cudaFuncSetAttribute(ln_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                max_dynamic_smem);
}

cudaError_t ln_persistent_occupancy(int dyn_smem, int *ctas_per_sm)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, ln_persistent_kernel, LN_T, dyn_smem);
}

cudaError_t ln_persistent_launch(const LnParams &p, int grid, int dyn_smem, cudaStream_t stream)
{
    LnParams args = p;
    void *kargs[] = {&args};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(ln_persistent_kernel), dim3(grid),
                                       dim3(LN_T), kargs, static_cast<size_t>(dyn_smem), stream);
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
