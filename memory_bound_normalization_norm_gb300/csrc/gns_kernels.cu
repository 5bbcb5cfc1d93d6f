// gns_kernels.cu - GroupNorm + LeakyReLU + x2 over contiguous segments.
//
// The operation is the GroupNorm page's (POPCORNBENCH transcript "Kimi-K2.6
// l2_p62": population mean and variance of each group, per-channel affine,
// LeakyReLU(t) = max(0,t) + slope*min(0,t), then x + x), taken to tensors
// with a spatial extent.  For x[N][C][S] (an NCHW tensor with S = H*W) the
// group g of sample n holds channels g*M .. g*M+M-1 (M = C/G) at every
// position: M*S values that are contiguous in memory.  So the tensor is R =
// N*G segments of L = M*S elements, and element e of segment r belongs to
// channel (r % G)*M + e/S.  The (N, C) form of the page is S = 1, L = M.
//
// Four kernels:
//  - register path: a segment is split over a thread-block cluster of CL
//    CTAs (CL = 1 for segments that fit one CTA).  Each CTA holds its slice
//    in registers, so x is read from HBM once and y written once.  The mean
//    (about the pivot x[r][0]) and then the exact M2 about the mean are
//    reduced over the CTA and then over the cluster through distributed
//    shared memory: every CTA publishes its partial in its own shared memory,
//    the cluster barrier orders it, and every warp reads the CL partials with
//    ld.shared::cluster and sums them in lane order, so all CTAs get the
//    same value.
//  - streamed register path (the same split, for slices of more than 256
//    vectors with 16-byte aligned rows; the automatic choice there): a
//    persistent grid of clusters walks segments, and each CTA's slice of the
//    next segment arrives by bulk copy (TMA engine, cp.async.bulk +
//    mbarrier) into a shared-memory buffer while the current one is reduced
//    and written from registers.  Each CTA reduces its slice to an exact
//    two-pass (mean, M2) and one all-to-all exchange per segment (st.async
//    into every CTA's shared memory, counted on that CTA's mbarrier) gives
//    every CTA the partials, merged with Chan's update in rank order.  A
//    cluster barrier with release semantics would wait for the CTA's
//    earlier y stores to drain (measured as the top stall, "membar"); the
//    mbarrier exchange does not.  bf16 slices stay packed in registers, so a
//    CTA holds twice as many vectors.  Every wait is bounded; see the
//    kernel.  Without the LeakyReLU x2 epilogue the same kernel is the
//    LayerNorm of rows of up to 131,072 elements (one group per row,
//    per-element gamma/beta).
//  - split path (segments longer than a 16-CTA cluster holds, or unaligned
//    vectors): the LayerNorm split path's statistics kernel writes one
//    (n, mean, M2, pivot) partial per (segment, chunk), and the apply kernel
//    here merges a segment's partials and applies, re-reading x.
//  - warp path: one warp per segment with scalar loads for short segments
//    that are not 4-element vectors (x re-read from L1).
#include <atomic>
#include <cstring>
#include <mutex>

#include "norm_internal.cuh"
#include <type_traits>

namespace normk {

namespace {

// ------------------------------------------------------------------ cluster helpers

__device__ __forceinline__ unsigned cluster_rank()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ unsigned cluster_id_x()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ unsigned cluster_count_x()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives; shared-memory writes
// before the arrive are visible to the cluster after the wait.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Load the float at `local` (this CTA's shared memory) from the same offset
// in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_peer_f32(const float *local, unsigned rank)
{
    const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(local));
    unsigned ra;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

// Cluster-wide sum of v (identical in all threads of a CTA): thread 0
// publishes it in `slot`, then each warp adds the cluster's CL values in
// lane order.  `slot` must not be rewritten until every CTA has passed the
// next cluster barrier.
__device__ __forceinline__ float cluster_sum(float v, float *slot, unsigned CL)
{
    if (threadIdx.x == 0)
        *slot = v;
    cluster_sync_all();
    const unsigned lane = threadIdx.x & 31;
    float t = lane < CL ? ld_peer_f32(slot, lane) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

// Address of `local` (this CTA's shared memory) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void *local, unsigned rank)
{
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
    return ra;
}

// Asynchronous 16-byte store into another CTA's shared memory whose arrival
// is counted (as transaction bytes) on that CTA's mbarrier.  Unlike a
// release at a cluster barrier it does not wait for this thread's earlier
// global stores.
__device__ __forceinline__ void st_async_f4(uint32_t remote, float4 v, uint32_t remote_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     remote),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
                 : "memory");
}

// One all-to-all exchange of the cluster's partial statistics: every CTA
// sends (mean, M2, flag, 0) of its slice into slot[rank] of every CTA
// (itself included), waits on its own `bar` (phase `parity`) for the CL
// slots, and merges them, rank j holding count_of(j) values, with Chan's
// pairwise update in a fixed order (the same result in every CTA).
// *flag_or gets the largest flag; *timed_out is set, for the whole CTA, if
// the wait gave up.
//
// A slot set and its mbarrier are reused two segments later.  A CTA sends
// into them only after it has received every CTA's exchange of the segment
// in between, which each CTA sends after it has read the set, so a send
// never overwrites unread values nor lands in the previous phase.
template <typename CountOf>
__device__ __forceinline__ Moments cluster_moments(float mean, float m2, float flag, float4 *slot, uint64_t *bar,
                                                   unsigned CL, unsigned rank, uint32_t parity, uint64_t wait_ns,
                                                   CountOf count_of, float *flag_or, bool *timed_out)
{
    if (threadIdx.x == 0)
        mbar_arrive_expect_tx(bar, CL * 16u);
    if (threadIdx.x < CL)
        st_async_f4(peer_addr(&slot[rank], threadIdx.x), make_float4(mean, m2, flag, 0.f),
                    peer_addr(bar, threadIdx.x));
    // one thread polls; the others wait at the CTA barrier without taking
    // issue slots, and see the slots through it
    const bool ok = threadIdx.x != 0 || mbar_wait_bounded(bar, parity, wait_ns);
    *timed_out = __syncthreads_or(!ok) != 0;
    const unsigned lane = threadIdx.x & 31;
    Moments m = {0.f, 0.f, 0.f};
    float f = 0.f;
    if (lane < CL) {
        const float4 w = slot[lane];
        m.n = count_of(lane);
        m.mean = w.x;
        m.m2 = w.y;
        f = w.z;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        f = fmaxf(f, __shfl_xor_sync(0xffffffffu, f, o));
    *flag_or = f;
    return warp_merge(m);
}

// ------------------------------------------------------------------ epilogue

__device__ __forceinline__ float lrelu_x2(float t, float slope)
{
    t = t > 0.f ? t : slope * t;
    return t + t;
}

__device__ __forceinline__ int64_t seg_div(int64_t e, int64_t S, bool narrow)
{
    return narrow ? static_cast<int64_t>(static_cast<uint32_t>(e) / static_cast<uint32_t>(S)) : e / S;
}

// How the four elements e .. e+3 (e a multiple of 4) map to channels.
enum AffineMode {
    AFF_ROW = 0,  // S == 1: four consecutive channels (one vector load)
    AFF_CHAN = 1, // S % 4 == 0: one channel
    AFF_ANY = 2,  // anything else: per element
};

__host__ __device__ constexpr int affine_mode(int64_t S)
{
    return S == 1 ? AFF_ROW : (S & 3) == 0 ? AFF_CHAN : AFF_ANY;
}

// gamma/beta of elements e .. e+3 of a segment whose first channel is cbase.
// cache: consecutive channels are read through L1 (worth it where every SM's
// CTAs read few distinct parts of gamma/beta), else with an L2 policy only.
template <typename T, int MODE>
__device__ __forceinline__ void seg_affine4(const T *gm, const T *bt, int64_t cbase, int64_t e, int64_t S,
                                            bool narrow, uint64_t pol, float4 &g, float4 &b, bool cache = false)
{
    if (MODE == AFF_ROW) {
        if (cache) {
            g = gm ? Io<T>::ld4_param(gm + cbase + e) : make_float4(1.f, 1.f, 1.f, 1.f);
            b = bt ? Io<T>::ld4_param(bt + cbase + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            g = gm ? Io<T>::ld4_ro(gm + cbase + e, pol) : make_float4(1.f, 1.f, 1.f, 1.f);
            b = bt ? Io<T>::ld4_ro(bt + cbase + e, pol) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    } else if (MODE == AFF_CHAN) {
        const int64_t c = cbase + seg_div(e, S, narrow);
        const float gv = gm ? Io<T>::ld1(gm + c) : 1.f, bv = bt ? Io<T>::ld1(bt + c) : 0.f;
        g = make_float4(gv, gv, gv, gv);
        b = make_float4(bv, bv, bv, bv);
    } else {
        float gv[4], bv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t c = cbase + seg_div(e + k, S, narrow);
            gv[k] = gm ? Io<T>::ld1(gm + c) : 1.f;
            bv[k] = bt ? Io<T>::ld1(bt + c) : 0.f;
        }
        g = make_float4(gv[0], gv[1], gv[2], gv[3]);
        b = make_float4(bv[0], bv[1], bv[2], bv[3]);
    }
}

__device__ __forceinline__ float4 gn_apply4(float4 v, const RowMean &rm, float4 g, float4 b, float slope)
{
    float4 t = ln_apply4(v, rm, g, b);
    t.x = lrelu_x2(t.x, slope);
    t.y = lrelu_x2(t.y, slope);
    t.z = lrelu_x2(t.z, slope);
    t.w = lrelu_x2(t.w, slope);
    return t;
}

// ------------------------------------------------------------------ register path

// grid: clusters of CL CTAs (CL = p.parts), each cluster walks segments
// r = cluster id, + cluster count, ...; CTA `rank` of a cluster owns vectors
// [rank*per, rank*per + per) of every segment it visits.
template <typename T, int NT, int V, int MODE>
__global__ void __launch_bounds__(NT) gns_reg_kernel(GnSegParams p)
{
    __shared__ float red[2][NT / 32];
    __shared__ float xch[2];
    const int tid = threadIdx.x;
    const unsigned CL = static_cast<unsigned>(p.parts);
    const bool clustered = CL > 1;
    const unsigned rank = clustered ? cluster_rank() : 0u;
    const int64_t cid = clustered ? cluster_id_x() : blockIdx.x;
    const int64_t ncl = clustered ? cluster_count_x() : gridDim.x;
    const int64_t L4 = p.seg_len >> 2;
    const int64_t per = small_ceil_div(L4, CL);
    const int64_t lo = per * rank;
    const int64_t n4 = lo < L4 ? (L4 - lo < per ? L4 - lo : per) : 0;
    const float Lf = static_cast<float>(p.seg_len);
    const float invL = 1.f / Lf; // the means below are products, not divisions
    constexpr bool narrow = true; // segments here are at most 16 * NT * V * 4 elements
    const T *x = static_cast<const T *>(p.x);
    T *y = static_cast<T *>(p.y);
    const T *gm = static_cast<const T *>(p.gamma);
    const T *bt = static_cast<const T *>(p.beta);
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    for (int64_t r = cid; r < p.rows; r += ncl) {
        const T *xr = x + r * p.seg_len;
        float4 v[V];
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t i = tid + k * NT;
            v[k] = i < n4 ? Io<T>::ld4_stream(xr + 4 * (lo + i), pol_stream) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // Every CTA of the cluster reads the pivot before the first cluster
        // barrier and stores only after the second, so y == x is safe.
        const float K = Io<T>::ld1(xr);
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            if (tid + k * NT < n4)
                s += ((v[k].x - K) + (v[k].y - K)) + ((v[k].z - K) + (v[k].w - K));
        }
        s = block_sum<NT>(s, red[0]);
        if (clustered)
            s = cluster_sum(s, &xch[0], CL);
        Moments tot;
        tot.n = Lf;
        tot.mean = s * invL;
        tot.m2 = 0.f;
        RowMean rm = finish_row(K, tot, p.eps);
        float q = 0.f;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            if (tid + k * NT < n4) {
                const float a = (v[k].x - rm.hi) - rm.lo, b = (v[k].y - rm.hi) - rm.lo;
                const float c = (v[k].z - rm.hi) - rm.lo, d = (v[k].w - rm.hi) - rm.lo;
                q += (a * a + b * b) + (c * c + d * d);
            }
        }
        q = block_sum<NT>(q, red[1]);
        if (clustered)
            q = cluster_sum(q, &xch[1], CL);
        rm.rstd = rsqrtf(fmaxf(q * invL, 0.f) + p.eps);
        const int64_t cbase = small_mod(r, p.G) * p.M;
        T *yr = y + r * p.seg_len;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t i = tid + k * NT;
            if (i < n4) {
                const int64_t e = 4 * (lo + i);
                float4 g, b;
                seg_affine4<T, MODE>(gm, bt, cbase, e, p.S, narrow, pol_keep, g, b);
                Io<T>::st4_stream(yr + e, gn_apply4(v[k], rm, g, b, p.slope), pol_stream);
            }
        }
    }
    // no CTA may exit while a peer can still read its partials
    if (clustered)
        cluster_sync_all();
}

// ------------------------------------------------------------------ streamed register path

// One slice buffer per CTA and registers sized for 4 CTAs per SM (a few
// spilled bytes at 8 vectors a thread) measured faster than two buffers at 3
// CTAs per SM: more clusters are resident, so the last wave of segments is
// shorter (GroupNorm (8,512,64,64): 29.6 vs 30.9 us; LayerNorm rows of
// 131,072: 112 vs 136 us).
constexpr int GNS_NBUF = 1;     // shared-memory slice buffers per CTA
constexpr int GNS_MIN_CTAS = 4; // CTAs per SM the register budget is sized for

template <typename T>
__device__ __forceinline__ float4 ld4_smem(const T *p);

template <>
__device__ __forceinline__ float4 ld4_smem<float>(const float *p)
{
    return *reinterpret_cast<const float4 *>(p);
}

template <typename T>
__device__ __forceinline__ float first_elem(const float4 &raw)
{
    if constexpr (sizeof(T) == 4)
        return raw.x;
    else
        return Io<__nv_bfloat16>::unpack(__float_as_uint(raw.x), 0u).x;
}

// A thread's copy of one 4-element vector of its slice, read as two float2
// pairs for the packed (f32x2) arithmetic.  fp32: d = x - K.  bf16: the
// packed values as loaded (two registers, so a CTA holds twice as many
// vectors), widened and shifted by `off` in one mixed-precision add a value
// where used; for fp32 `off` is added to d.
template <typename T>
struct Held;

template <>
struct Held<float> {
    float2 lo, hi;
    __device__ __forceinline__ void clear() { lo = hi = make_float2(0.f, 0.f); }
    __device__ __forceinline__ void load(const float *p, float K)
    {
        const float4 x = ld4_smem<float>(p);
        const float2 nk = make_float2(-K, -K);
        lo = __fadd2_rn(make_float2(x.x, x.y), nk);
        hi = __fadd2_rn(make_float2(x.z, x.w), nk);
    }
    // d (+ off for a nonzero off)
    __device__ __forceinline__ void pair(float2 off, bool add, float2 &l, float2 &h) const
    {
        l = add ? __fadd2_rn(lo, off) : lo;
        h = add ? __fadd2_rn(hi, off) : hi;
    }
};

template <>
struct Held<__nv_bfloat16> {
    uint2 raw;
    __device__ __forceinline__ void clear() { raw = make_uint2(0u, 0u); }
    __device__ __forceinline__ void load(const __nv_bfloat16 *p, float) { raw = *reinterpret_cast<const uint2 *>(p); }
    // x + off (off = -K for d), widened again in each pass
    __device__ __forceinline__ void pair(float2 off, bool, float2 &l, float2 &h) const
    {
        l = bf16x2_add(raw.x, off);
        h = bf16x2_add(raw.y, off);
    }
};

// LeakyReLU of a pair: max(t, slope t) for slope <= 1 (negative slopes too)
// and min(t, slope t) for slope > 1 are t > 0 ? t : slope t.
__device__ __forceinline__ float2 lrelu2(float2 t, float2 slope2, bool steep)
{
    const float2 u = __fmul2_rn(t, slope2);
    return steep ? make_float2(fminf(t.x, u.x), fminf(t.y, u.y)) : make_float2(fmaxf(t.x, u.x), fmaxf(t.y, u.y));
}

// grid: a persistent set of clusters of CL = p.parts CTAs (CL = 1 allowed);
// cluster c walks segments r_k = c + k * (cluster count).  CTA `rank` owns
// vectors [rank * per, rank * per + per) of each segment (per = p.per4).
// Dynamic shared memory: GNS_NBUF slice buffers of per vectors; a slice
// moves to registers as soon as it lands and the buffer is refilled at once,
// so the next segment's slice is in flight while the current one is reduced
// and written.  Per segment each CTA computes the exact two-pass (mean, M2) of
// its slice about the pivot, and one all-to-all exchange (st.async into
// every CTA's shared memory, counted on its mbarrier) gives every CTA the
// CL partials, merged in rank order.
//
// Failure handling: a CTA whose bulk-copy wait gives up flags its partials
// from then on; every CTA sees a flag in the same exchange, so from that
// segment on the whole cluster writes nothing, stops waiting for copies and
// keeps exchanging (the exchanges still complete) until the end; each CTA
// then drains its own copies.
template <typename T, int NT, int V, int MODE, bool ACT, int MINB>
__global__ void __launch_bounds__(NT, MINB) gns_stream_kernel(GnSegParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(16) float4 piv[2]; // first 16 bytes of the segment, copied with the slice
    __shared__ __align__(8) uint64_t full[2];
    __shared__ __align__(8) uint64_t xbar[2];     // exchange, per segment parity
    __shared__ __align__(16) float4 xslot[2][16]; // (mean, M2, flag, 0) per rank
    __shared__ float red[2][NT / 32];
    const int tid = threadIdx.x;
    const unsigned CL = static_cast<unsigned>(p.parts);
    const bool clustered = CL > 1;
    const unsigned rank = clustered ? cluster_rank() : 0u;
    const int64_t cid = clustered ? cluster_id_x() : blockIdx.x;
    const int64_t ncl = clustered ? cluster_count_x() : gridDim.x;
    const int64_t L4 = p.seg_len >> 2;
    const int per = p.per4;
    const int64_t lo = static_cast<int64_t>(per) * rank;
    const int n4 = lo < L4 ? static_cast<int>(L4 - lo < per ? L4 - lo : per) : 0;
    const float nloc = 4.f * static_cast<float>(n4);
    // values held by rank j
    const auto count_of = [L4, per](unsigned j) {
        const int64_t l = static_cast<int64_t>(per) * j;
        return l < L4 ? 4.f * static_cast<float>(L4 - l < per ? L4 - l : per) : 0.f;
    };
    const uint32_t slice_bytes = static_cast<uint32_t>(n4) * 4u * sizeof(T);
    T *buf0 = reinterpret_cast<T *>(smem);
    T *buf1 = GNS_NBUF > 1 ? buf0 + static_cast<size_t>(per) * 4 : buf0;
    constexpr bool narrow = true;
    const T *x = static_cast<const T *>(p.x);
    T *y = static_cast<T *>(p.y);
    const T *gm = static_cast<const T *>(p.gamma);
    const T *bt = static_cast<const T *>(p.beta);
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    // segments of this cluster (32-bit division when the counts fit)
    int64_t nk = 0;
    if (cid < p.rows) {
        const int64_t num = p.rows - cid + ncl - 1;
        nk = num <= 0xffffffffll ? static_cast<int64_t>(static_cast<uint32_t>(num) / static_cast<uint32_t>(ncl))
                                 : num / ncl;
    }
    // group of segment cid + k * ncl, stepped by ncl mod G per segment
    int64_t gcur = small_mod(cid, p.G);
    const int64_t gstep = small_mod(ncl, p.G);
    const uint64_t xwait_ns = p.timeout_ns > 100000000ull ? p.timeout_ns : 100000000ull;
    // With one channel per vector, the channel of this thread's vector j
    // within a segment is the same for every segment: c0 and r0 are those of
    // vector 0 (quotient and remainder of its first element by S); vector
    // j + 1 starts 4 * NT elements further on, qstep channels and rstep
    // elements on.
    const uint32_t S32 = static_cast<uint32_t>(p.S);
    const uint32_t e0 = static_cast<uint32_t>(4 * (lo + tid));
    const uint32_t c0 = MODE == AFF_CHAN ? e0 / S32 : 0u, r0 = MODE == AFF_CHAN ? e0 % S32 : 0u;
    const uint32_t qstep = MODE == AFF_CHAN ? (4u * NT) / S32 : 0u, rstep = MODE == AFF_CHAN ? (4u * NT) % S32 : 0u;

    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        fence_mbar_init();
    }
    // every CTA's barriers are initialized before any CTA sends to them
    if (clustered)
        cluster_sync_all();
    else
        __syncthreads();
    // Launched with programmatic stream serialization (the GroupNorm form):
    // wait for the previous kernel of the stream before the first global
    // access.  Without that launch attribute this returns at once.
    pdl_wait();
    // thread 0: copy this CTA's slice of segment k (and the segment's first
    // 16 bytes, which hold the pivot) into buffer k & 1
    auto issue = [&](int64_t k) {
        const int b = static_cast<int>(k % GNS_NBUF);
        const T *xr = x + (cid + k * ncl) * p.seg_len;
        mbar_arrive_expect_tx(&full[b], slice_bytes + 16u);
        bulk_g2s(&piv[b], xr, 16u, &full[b], pol_stream);
        if (slice_bytes)
            bulk_g2s(b ? buf1 : buf0, xr + 4 * lo, slice_bytes, &full[b], pol_stream);
    };
    int64_t issued = 0;
    if (tid == 0) {
        for (; issued < GNS_NBUF && issued < nk; ++issued)
            issue(issued);
    }
    bool stopped = false; // this cluster writes nothing more
    bool gave_up = false; // this CTA's own wait gave up
    int64_t consumed = 0; // segments whose copies this CTA has seen complete
    for (int64_t k = 0; k < nk; ++k) {
        const int b = static_cast<int>(k & 1); // exchange slots: segment parity
        const uint32_t par = static_cast<uint32_t>((k >> 1) & 1);
        const int db = static_cast<int>(k % GNS_NBUF); // data buffer
        const uint32_t dpar = static_cast<uint32_t>((k / GNS_NBUF) & 1);
        if (!stopped) {
            // one thread polls, the others wait at the CTA barrier; the
            // decision is the whole CTA's
            const bool ok = tid != 0 || mbar_wait_bounded(&full[db], dpar, p.timeout_ns);
            if (__syncthreads_or(!ok)) {
                gave_up = true;
                stopped = true;
            } else {
                consumed = k + 1;
            }
        }
        const T *sb = db ? buf1 : buf0;
        // FAST: this CTA's slice fills every thread's V vectors, and (for
        // one channel a vector) a step of 4 * NT elements crosses at most one
        // channel boundary; then no vector needs a range check
        auto seg = [&](auto fast_c) {
            constexpr bool FAST = decltype(fast_c)::value;
            Held<T> v[V];
            float K = 0.f;
#pragma unroll
            for (int j = 0; j < V; ++j)
                v[j].clear();
            if (!stopped) {
                K = first_elem<T>(piv[db]);
                const T *st = sb + 4 * tid;
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    if (FAST || tid + j * NT < n4)
                        v[j].load(st + 4 * NT * j, K);
                }
            }
            // exact two-pass statistics of this CTA's slice about the pivot, in
            // f32x2 pairs
            constexpr bool bf = sizeof(T) == 2;
            const float2 negk = make_float2(-K, -K); // bf16: d = x - K as it is widened
            float2 sl = make_float2(0.f, 0.f), sh = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < V; ++j) {
                if (FAST || tid + j * NT < n4) {
                    float2 l, h;
                    v[j].pair(negk, false, l, h);
                    sl = __fadd2_rn(sl, l);
                    sh = __fadd2_rn(sh, h);
                }
            }
            float s = (sl.x + sl.y) + (sh.x + sh.y);
            s = block_sum<NT>(s, red[0]);
            // every thread has its values in registers: refill this buffer with
            // the segment GNS_NBUF ahead
            if (tid == 0 && !stopped && issued < nk && issued == k + GNS_NBUF) {
                fence_proxy_async_smem();
                issue(issued);
                ++issued;
            }
            const float mloc = n4 ? s / nloc : 0.f;
            // deviations from the slice mean: d - mloc (fp32), or x - (K + mloc)
            // with the centre rounded once (bf16; its offset from the exact
            // centre adds at most n * ulp(K)^2 / 4 to M2)
            const float2 nc = bf ? make_float2(-(K + mloc), -(K + mloc)) : make_float2(-mloc, -mloc);
            float2 ql = make_float2(0.f, 0.f), qh = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < V; ++j) {
                if (FAST || tid + j * NT < n4) {
                    float2 l, h;
                    v[j].pair(nc, true, l, h);
                    ql = __ffma2_rn(l, l, ql);
                    qh = __ffma2_rn(h, h, qh);
                }
            }
            float q = (ql.x + ql.y) + (qh.x + qh.y);
            q = block_sum<NT>(q, red[1]);
            Moments tot;
            tot.n = nloc;
            tot.mean = mloc;
            tot.m2 = q;
            if (clustered) {
                // a stopped CTA's partial is flagged, so no CTA uses it
                float f = 0.f;
                bool to = false;
                tot = cluster_moments(mloc, q, stopped ? 1.f : 0.f, xslot[b], &xbar[b], CL, rank, par, xwait_ns,
                                      count_of, &f, &to);
                if (f != 0.f || to)
                    stopped = true;
            }
            // the last segment's statistics are merged: the next kernel of the
            // stream may be scheduled onto SMs as this grid's CTAs finish
            if (k == nk - 1)
                pdl_trigger();
            if (stopped)
                return; // keep exchanging, write nothing
            // ACT: y = 2 * LReLU((x - mean) * rstd * gamma + beta), with x - mean
            // = d - tot.mean; LReLU is positively homogeneous, so the factor 2
            // goes into the affine map: 2t = d * a + c, a = 2 * rstd * gamma,
            // c = 2 * beta - tot.mean * a.  Without ACT (LayerNorm): y = d * a + c
            // with a = rstd * gamma, c = beta - tot.mean * a.  Pairs in f32x2.
            const float rstd = rsqrtf(fmaxf(tot.m2 / tot.n, 0.f) + p.eps);
            const float mean_d = tot.mean;
            const float2 slope2 = make_float2(p.slope, p.slope);
            const bool steep = p.slope > 1.f;
            constexpr float sc = ACT ? 2.f : 1.f;
            const float sr = sc * rstd;
            const int64_t r = cid + k * ncl;
            const int64_t cbase = gcur * p.M;
            T *yr = y + r * p.seg_len;
            T *yt = yr + 4 * (lo + tid); // this thread's vector 0
            uint32_t cj = c0, rj = r0;  // channel of vector j within the segment, and the remainder
            uint32_t cur = 0xffffffffu; // the channel a2 / c2 belong to
            float2 a2 = make_float2(0.f, 0.f), c2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int i = tid + j * NT;
                if (FAST || i < n4) {
                    const int64_t e = 4 * (lo + i);
                    float2 l, h;
                    v[j].pair(negk, false, l, h);
                    if constexpr (MODE == AFF_CHAN) {
                        if (cj != cur) {
                            // a new channel: its gamma/beta (each run of a
                            // thread's vectors in one channel loads them once)
                            cur = cj;
                            const int64_t c = cbase + cj;
                            const float gv = gm ? Io<T>::ld1(gm + c) : 1.f, bv = bt ? Io<T>::ld1(bt + c) : 0.f;
                            const float a = sr * gv;
                            a2 = make_float2(a, a);
                            const float cc = fmaf(-mean_d, a, sc * bv);
                            c2 = make_float2(cc, cc);
                        }
                        l = __ffma2_rn(l, a2, c2);
                        h = __ffma2_rn(h, a2, c2);
                    } else {
                        float4 g, bb;
                        seg_affine4<T, MODE>(gm, bt, cbase, e, p.S, narrow, pol_keep, g, bb, p.cache_gb != 0);
                        const float2 sr2 = make_float2(sr, sr), nm = make_float2(-mean_d, -mean_d);
                        const float2 al = __fmul2_rn(make_float2(g.x, g.y), sr2);
                        const float2 ah = __fmul2_rn(make_float2(g.z, g.w), sr2);
                        float2 bl = make_float2(bb.x, bb.y), bh = make_float2(bb.z, bb.w);
                        if constexpr (ACT) {
                            bl = __fadd2_rn(bl, bl);
                            bh = __fadd2_rn(bh, bh);
                        }
                        l = __ffma2_rn(l, al, __ffma2_rn(nm, al, bl));
                        h = __ffma2_rn(h, ah, __ffma2_rn(nm, ah, bh));
                    }
                    if constexpr (ACT) {
                        l = lrelu2(l, slope2, steep);
                        h = lrelu2(h, slope2, steep);
                    }
                    Io<T>::st4_stream(yt + 4 * NT * j, make_float4(l.x, l.y, h.x, h.y), pol_stream);
                }
                if constexpr (MODE == AFF_CHAN) {
                    // S % 4 == 0: a step of 4 * NT elements is qstep whole
                    // channels (none when S >= 4 * NT) and rstep elements,
                    // which cross at most one more channel boundary
                    if (FAST) {
                        rj += 4u * NT;
                    } else {
                        rj += rstep;
                        cj += qstep;
                    }
                    if (rj >= S32) {
                        rj -= S32;
                        ++cj;
                    }
                }
            }
        };
        if (n4 == NT * V && (MODE != AFF_CHAN || S32 >= 4u * NT))
            seg(std::true_type{});
        else
            seg(std::false_type{});
        gcur += gstep;
        if (gcur >= p.G)
            gcur -= p.G;
    }
    if (stopped && tid == 0) {
        if (gave_up)
            record_error(p.err, NORM_ERR_TIMEOUT);
        // the copies this CTA issued and never saw complete still write its
        // shared memory: wait for them before the CTA exits
        for (int64_t j = consumed; j < issued; ++j)
            mbar_wait_bounded(&full[j % GNS_NBUF], static_cast<uint32_t>((j / GNS_NBUF) & 1), xwait_ns);
    }
}

// ------------------------------------------------------------------ split path: apply

constexpr int GS_T = 256;

template <typename T, bool VEC>
__global__ void __launch_bounds__(GS_T) gns_split_apply_kernel(GnSegParams p)
{
    pdl_begin();
    __shared__ RowMean row_mean;
    const int P = p.parts;
    const bool narrow = p.seg_len <= int64_t(0xffffffff);
    const T *x = static_cast<const T *>(p.x);
    T *y = static_cast<T *>(p.y);
    const T *gm = static_cast<const T *>(p.gamma);
    const T *bt = static_cast<const T *>(p.beta);
    // Segments and chunks in the reverse of the statistics kernel's order:
    // the most recently read part of x is the likeliest still in L2.
    for (int64_t rr = blockIdx.y; rr < p.rows; rr += gridDim.y) {
        const int64_t r = p.rows - 1 - rr;
        const int pc = P - 1 - static_cast<int>(blockIdx.x);
        const T *xr = x + r * p.seg_len;
        T *yr = y + r * p.seg_len;
        if (threadIdx.x < 32) {
            const float K = ld_l2_f4(p.part + r * P).w;
            const Moments tot = merge_partials_warp(p.part + r * P, P, K);
            if (threadIdx.x == 0)
                row_mean = finish_row(K, tot, p.eps);
        }
        __syncthreads();
        const RowMean rm = row_mean;
        const int64_t cbase = small_mod(r, p.G) * p.M;
        const int64_t lo = static_cast<int64_t>(pc) * p.chunk;
        const int64_t hi = (lo + p.chunk < p.seg_len) ? lo + p.chunk : p.seg_len;
        if (VEC) {
            const uint64_t pol = policy_evict_first();
            const uint64_t pol_gb = policy_evict_last();
            const int mode = affine_mode(p.S);
            auto one = [&](int64_t i, const float4 &q) {
                float4 g, b;
                switch (mode) {
                case AFF_ROW: seg_affine4<T, AFF_ROW>(gm, bt, cbase, 4 * i, p.S, narrow, pol_gb, g, b); break;
                case AFF_CHAN: seg_affine4<T, AFF_CHAN>(gm, bt, cbase, 4 * i, p.S, narrow, pol_gb, g, b); break;
                default: seg_affine4<T, AFF_ANY>(gm, bt, cbase, 4 * i, p.S, narrow, pol_gb, g, b); break;
                }
                Io<T>::st4_stream(yr + 4 * i, gn_apply4(q, rm, g, b, p.slope), pol);
            };
            int64_t i = lo / 4 + threadIdx.x;
            const int64_t e4 = hi / 4;
            // four loads of x in flight per thread
            for (; i + 3 * GS_T < e4; i += 4 * GS_T) {
                float4 q[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    q[u] = Io<T>::ld4_stream(xr + 4 * (i + u * GS_T), pol);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    one(i + u * GS_T, q[u]);
            }
            for (; i < e4; i += GS_T)
                one(i, Io<T>::ld4_stream(xr + 4 * i, pol));
        } else {
            for (int64_t i = lo + threadIdx.x; i < hi; i += GS_T) {
                const int64_t c = cbase + seg_div(i, p.S, narrow);
                const float g = gm ? Io<T>::ld1(gm + c) : 1.f;
                const float b = bt ? Io<T>::ld1(bt + c) : 0.f;
                const float t = fmaf(((Io<T>::ld1(xr + i) - rm.hi) - rm.lo) * rm.rstd, g, b);
                Io<T>::st1(yr + i, lrelu_x2(t, p.slope));
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ team path

// Short segments (at most 256 items, an item being E = 4, 2 or 1 consecutive
// elements): a team of T = 2^tlog lanes owns one segment, lane j of the team
// holding items j, j + T, ..., j + (W - 1) T (W <= WMAX, guarded at the
// segment's end).  T is the narrowest team that gives each lane at most
// TEAM_TARGET_W items (up to a full warp): wider teams spend more shuffles
// per element, narrower ones more registers (a group of 48 channels is 4
// lanes x 3 vectors).  32 / T segments per warp, 8 warps a CTA, grid-stride
// over segments.  The mean about the pivot (the segment's first element) and
// then M2 about the mean are reduced with xor shuffles within the team: no
// CTA barrier.  Teams of a warp may leave the loop at different times;
// shuffles name only the team's lanes.
constexpr int TEAM_W = 8;
constexpr int TEAM_TARGET_W = 4;

template <int E>
__device__ __forceinline__ float comp(const float4 &v, int k)
{
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

template <typename T, int E>
__device__ __forceinline__ float4 team_load(const T *p, uint64_t pol)
{
    if constexpr (E == 4)
        return Io<T>::ld4_stream(p, pol);
    if constexpr (E == 2) {
        const float2 t = Io<T>::ld2_stream(p, pol);
        return make_float4(t.x, t.y, 0.f, 0.f);
    }
    return make_float4(Io<T>::ld1_stream(p, pol), 0.f, 0.f, 0.f);
}

template <typename T, int E>
__device__ __forceinline__ void team_store(T *p, const float4 &o, uint64_t pol)
{
    if constexpr (E == 4)
        Io<T>::st4_stream(p, o, pol);
    else if constexpr (E == 2)
        Io<T>::st2_stream(p, make_float2(o.x, o.y), pol);
    else
        Io<T>::st1_stream(p, o.x, pol);
}

// Threads of a team-kernel CTA: 128 for 4-element items, 256 otherwise.
// Measured on GB300, each build timed alone (us, 256 -> 128 threads): groups
// of 48 (8192, 1536) fp32 20.7 -> 19.4, bf16 18.7 -> 17.6; of 96 20.7 -> 19.5;
// of 192 fp32 38.0 -> 35.1; pairs (groups of 30, fp32) 39.6 -> 41.0.
template <int E>
constexpr int team_threads()
{
    return E == 4 ? 128 : 256;
}

template <typename T, int E, int MODE, int WMAX>
__global__ void __launch_bounds__(team_threads<E>()) gns_team_kernel(GnSegParams p, int tlog, int W)
{
    pdl_begin();
    const int Tn = 1 << tlog;
    const int lane = threadIdx.x & 31;
    const int j = lane & (Tn - 1);
    const int first = lane & ~(Tn - 1);
    const unsigned tmask = Tn == 32 ? 0xffffffffu : (((1u << Tn) - 1u) << first);
    const int64_t teams_per_cta = blockDim.x >> tlog;
    const int64_t nteams = static_cast<int64_t>(gridDim.x) * teams_per_cta;
    const int items = static_cast<int>(p.seg_len / E);
    // 1 / L once: the means below are products, not divisions
    const float invL = 1.f / static_cast<float>(p.seg_len);
    // which of this lane's item slots hold an item: the same in every segment
    bool in[WMAX];
#pragma unroll
    for (int w = 0; w < WMAX; ++w)
        in[w] = w < W && j + w * Tn < items;
    const T *x = static_cast<const T *>(p.x);
    T *y = static_cast<T *>(p.y);
    const T *gm = static_cast<const T *>(p.gamma);
    const T *bt = static_cast<const T *>(p.beta);
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    const float slope = p.slope;
    int64_t r = static_cast<int64_t>(blockIdx.x) * teams_per_cta + (threadIdx.x >> tlog);
    // group index (r mod G) of the current segment, stepped without a
    // division per segment
    int64_t rg = r % p.G;
    const int64_t rg_step = nteams % p.G;
    const float2 slope2 = make_float2(slope, slope);
    const bool steep = slope > 1.f;
    // fp32: x of this team's next segment is loaded while the current one is
    // reduced and written (another segment, so y == x is safe), doubling the
    // bytes in flight.  bf16 loads widen as they arrive, which would stall
    // right behind the prefetch: measured slower, so bf16 loads in turn.
    constexpr bool PF = sizeof(T) == 4;
    float4 nx[PF ? WMAX : 1];
    // this lane's first item of segment r, in x and in y, stepped by
    // nteams segments a loop
    const int64_t seg_step = nteams * p.seg_len;
    const T *xl = x + r * p.seg_len + E * j;
    T *yl = y + r * p.seg_len + E * j;
    auto load_seg = [&](int64_t rr, const T *src, float4 *dst) {
#pragma unroll
        for (int w = 0; w < WMAX; ++w)
            dst[w] = (in[w] && rr < p.rows) ? team_load<T, E>(src + E * w * Tn, pol_stream)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    if constexpr (PF)
        load_seg(r, xl, nx);
    for (; r < p.rows; r += nteams, xl += seg_step, yl += seg_step) {
        float4 v[WMAX];
        if constexpr (PF) {
#pragma unroll
            for (int w = 0; w < WMAX; ++w)
                v[w] = nx[w];
            load_seg(r + nteams, xl + seg_step, nx);
        } else {
            load_seg(r, xl, v);
        }
        // the segment's first element, from the team's first lane; every
        // lane reads it before any lane of the team stores (the shuffles
        // below order them), so y == x is safe.  From here on v holds
        // d = x - K.
        const float K = __shfl_sync(tmask, v[0].x, first);
        float s = 0.f;
        if constexpr (E == 4) {
            // four-element items: the arithmetic in f32x2 pairs
            const float2 negk = make_float2(-K, -K);
            float2 sp = make_float2(0.f, 0.f);
#pragma unroll
            for (int w = 0; w < WMAX; ++w) {
                if (in[w]) {
                    const float2 l = __fadd2_rn(make_float2(v[w].x, v[w].y), negk);
                    const float2 h = __fadd2_rn(make_float2(v[w].z, v[w].w), negk);
                    v[w] = make_float4(l.x, l.y, h.x, h.y);
                    sp = __fadd2_rn(sp, __fadd2_rn(l, h));
                }
            }
            s = sp.x + sp.y;
        } else {
#pragma unroll
            for (int w = 0; w < WMAX; ++w) {
                if (in[w]) {
                    v[w].x -= K;
                    if constexpr (E == 2) {
                        v[w].y -= K;
                        s += v[w].x + v[w].y;
                    } else {
                        s += v[w].x;
                    }
                }
            }
        }
        for (int o = Tn >> 1; o > 0; o >>= 1)
            s += __shfl_xor_sync(tmask, s, o);
        const float mean_d = s * invL;
        float q = 0.f;
        if constexpr (E == 4) {
            const float2 nm = make_float2(-mean_d, -mean_d);
            float2 qp = make_float2(0.f, 0.f);
#pragma unroll
            for (int w = 0; w < WMAX; ++w) {
                if (in[w]) {
                    const float2 l = __fadd2_rn(make_float2(v[w].x, v[w].y), nm);
                    const float2 h = __fadd2_rn(make_float2(v[w].z, v[w].w), nm);
                    qp = __ffma2_rn(h, h, __ffma2_rn(l, l, qp));
                }
            }
            q = qp.x + qp.y;
        } else {
#pragma unroll
            for (int w = 0; w < WMAX; ++w) {
                if (in[w]) {
#pragma unroll
                    for (int k = 0; k < E; ++k) {
                        const float a = comp<E>(v[w], k) - mean_d;
                        q = fmaf(a, a, q);
                    }
                }
            }
        }
        for (int o = Tn >> 1; o > 0; o >>= 1)
            q += __shfl_xor_sync(tmask, q, o);
        // 2 LeakyReLU(t) = LeakyReLU(2 t), and 2 t = d * sc + c with
        // sc = 2 rstd gamma, c = 2 beta - mean_d * sc: one FMA an element
        const float rstd2 = 2.f * rsqrtf(fmaxf(q * invL, 0.f) + p.eps);
        const int64_t cbase = rg * p.M;
#pragma unroll
        for (int w = 0; w < WMAX; ++w) {
            if (!in[w])
                continue;
            const int i = j + w * Tn;
            if constexpr (E == 4) {
                float4 g4, b4;
                seg_affine4<T, MODE>(gm, bt, cbase, int64_t(4) * i, p.S, true, pol_keep, g4, b4, p.cache_gb != 0);
                const float2 r2 = make_float2(rstd2, rstd2), nm = make_float2(-mean_d, -mean_d);
                const float2 al = __fmul2_rn(make_float2(g4.x, g4.y), r2), ah = __fmul2_rn(make_float2(g4.z, g4.w), r2);
                const float2 bl = make_float2(b4.x, b4.y), bh = make_float2(b4.z, b4.w);
                float2 tl = __ffma2_rn(make_float2(v[w].x, v[w].y), al, __ffma2_rn(nm, al, __fadd2_rn(bl, bl)));
                float2 th = __ffma2_rn(make_float2(v[w].z, v[w].w), ah, __ffma2_rn(nm, ah, __fadd2_rn(bh, bh)));
                tl = lrelu2(tl, slope2, steep);
                th = lrelu2(th, slope2, steep);
                team_store<T, E>(yl + E * w * Tn, make_float4(tl.x, tl.y, th.x, th.y), pol_stream);
            } else {
                float g[4], b[4];
#pragma unroll
                for (int k = 0; k < E; ++k) {
                    const int e = E * i + k;
                    const int64_t c = cbase + (MODE == AFF_ROW ? int64_t(e) : seg_div(e, p.S, true));
                    g[k] = gm ? Io<T>::ld1(gm + c) : 1.f;
                    b[k] = bt ? Io<T>::ld1(bt + c) : 0.f;
                }
                float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int k = 0; k < E; ++k) {
                    const float sc = rstd2 * g[k];
                    const float t = fmaf(comp<E>(v[w], k), sc, fmaf(-mean_d, sc, b[k] + b[k]));
                    o[k] = t > 0.f ? t : slope * t;
                }
                team_store<T, E>(yl + E * w * Tn, make_float4(o[0], o[1], o[2], o[3]), pol_stream);
            }
        }
        rg += rg_step;
        if (rg >= p.G)
            rg -= p.G;
    }
}

// ------------------------------------------------------------------ warp path

// One warp per segment: mean, then M2 about the mean (a second read that
// hits L1/L2), then apply (a third).
template <typename T>
__global__ void __launch_bounds__(256) gns_warp_kernel(GnSegParams p)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const bool narrow = p.seg_len <= int64_t(0xffffffff);
    const float Lf = static_cast<float>(p.seg_len);
    const float invL = 1.f / Lf; // the means below are products, not divisions
    const T *x = static_cast<const T *>(p.x);
    T *y = static_cast<T *>(p.y);
    const T *gm = static_cast<const T *>(p.gamma);
    const T *bt = static_cast<const T *>(p.beta);
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < p.rows;
         r += warps) {
        const T *xr = x + r * p.seg_len;
        T *yr = y + r * p.seg_len;
        // the pivot keeps the sum small when |mean| >> std
        const float K = Io<T>::ld1(xr);
        float s = 0.f;
        for (int64_t j = lane; j < p.seg_len; j += 32)
            s += Io<T>::ld1(xr + j) - K;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            s += __shfl_xor_sync(0xffffffffu, s, o);
        Moments tot;
        tot.n = Lf;
        tot.mean = s * invL;
        tot.m2 = 0.f;
        RowMean rm = finish_row(K, tot, p.eps);
        float q = 0.f;
        for (int64_t j = lane; j < p.seg_len; j += 32) {
            const float d = (Io<T>::ld1(xr + j) - rm.hi) - rm.lo;
            q = fmaf(d, d, q);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            q += __shfl_xor_sync(0xffffffffu, q, o);
        rm.rstd = rsqrtf(fmaxf(q * invL, 0.f) + p.eps);
        const int64_t cbase = small_mod(r, p.G) * p.M;
        // every lane has read the whole segment (the shuffles above are
        // warp-wide), so with y == x the stores below are safe
        for (int64_t j = lane; j < p.seg_len; j += 32) {
            const int64_t c = cbase + seg_div(j, p.S, narrow);
            const float g = gm ? Io<T>::ld1(gm + c) : 1.f;
            const float b = bt ? Io<T>::ld1(bt + c) : 0.f;
            const float t = fmaf(((Io<T>::ld1(xr + j) - rm.hi) - rm.lo) * rm.rstd, g, b);
            Io<T>::st1(yr + j, lrelu_x2(t, p.slope));
        }
    }
}

// ------------------------------------------------------------------ register-path dispatch

constexpr int GNS_MAX_V = 8;
constexpr int GNS_MAX_NT = 256;
constexpr int GNS_MAX_CLUSTER = 16;

using RegKernel = void (*)(GnSegParams);

constexpr int GNS_VARIANTS = 18; // 6 CTA shapes x 3 affine modes

// Threads and vectors per thread for a CTA slice of `per` vectors: the
// smallest CTA that holds it with at most 4 (64 threads) or 8 vectors a
// thread, vectors a power of two.  *idx numbers the variant.
template <typename T, int MODE>
RegKernel reg_kernel_for(int64_t per, int *nt, int *idx)
{
    *nt = 0;
    *idx = -1;
    if (per <= 0 || per > 2048)
        return nullptr;
    if (per <= 64) {
        *nt = 64, *idx = 0;
        return gns_reg_kernel<T, 64, 1, MODE>;
    }
    if (per <= 128) {
        *nt = 64, *idx = 1;
        return gns_reg_kernel<T, 64, 2, MODE>;
    }
    if (per <= 256) {
        *nt = 64, *idx = 2;
        return gns_reg_kernel<T, 64, 4, MODE>;
    }
    if (per <= 512) {
        *nt = 128, *idx = 3;
        return gns_reg_kernel<T, 128, 4, MODE>;
    }
    if (per <= 1024) {
        *nt = 128, *idx = 4;
        return gns_reg_kernel<T, 128, 8, MODE>;
    }
    *nt = 256, *idx = 5;
    return gns_reg_kernel<T, 256, 8, MODE>;
}

template <typename T>
RegKernel reg_kernel_t(int64_t per, int mode, int *nt, int *idx)
{
    switch (mode) {
    case AFF_ROW: return reg_kernel_for<T, AFF_ROW>(per, nt, idx);
    case AFF_CHAN: return reg_kernel_for<T, AFF_CHAN>(per, nt, idx);
    default: return reg_kernel_for<T, AFF_ANY>(per, nt, idx);
    }
}

// The kernel for a segment of seg_len elements with S positions per channel
// over `cluster` CTAs; *idx numbers it among the variants of its dtype.
RegKernel reg_kernel(int64_t seg_len, int64_t S, bool bf16, int cluster, int *nt, int *idx)
{
    const int64_t L4 = seg_len / 4;
    const int64_t per = (L4 + cluster - 1) / cluster;
    const int mode = affine_mode(S);
    const RegKernel k = bf16 ? reg_kernel_t<__nv_bfloat16>(per, mode, nt, idx)
                             : reg_kernel_t<float>(per, mode, nt, idx);
    *idx += 6 * mode;
    return k;
}

void cluster_config(cudaLaunchConfig_t *cfg, cudaLaunchAttribute *attr, int nt, int cluster, unsigned grid,
                    cudaStream_t stream)
{
    std::memset(cfg, 0, sizeof(*cfg));
    cfg->gridDim = dim3(grid);
    cfg->blockDim = dim3(static_cast<unsigned>(nt));
    cfg->dynamicSmemBytes = 0;
    cfg->stream = stream;
    attr->id = cudaLaunchAttributeClusterDimension;
    attr->val.clusterDim.x = static_cast<unsigned>(cluster);
    attr->val.clusterDim.y = 1;
    attr->val.clusterDim.z = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
}

int log2_cluster(int cluster)
{
    int l = 0;
    while ((1 << l) < cluster)
        ++l;
    return l;
}

// Co-resident clusters per (device, dtype, variant, cluster size), queried
// once: -1 = not yet known.
constexpr int GNS_DEVICES = 64;
std::atomic<int> g_active[GNS_DEVICES][2][GNS_VARIANTS][5];
std::once_flag g_active_init;

cudaError_t query_active(RegKernel k, int nt, int cluster, int *clusters)
{
    *clusters = 0;
    if (cluster == 1) {
        int per_sm = 0, sms = 0, dev = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, nt, 0);
        if (e == cudaSuccess)
            e = cudaGetDevice(&dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        *clusters = per_sm * sms;
        return e;
    }
    if (cluster > 8) {
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess)
            return e;
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr;
    cluster_config(&cfg, &attr, nt, cluster, static_cast<unsigned>(cluster), 0);
    return cudaOccupancyMaxActiveClusters(clusters, k, &cfg);
}

} // namespace

int64_t gns_reg_capacity4(int cluster)
{
    return int64_t(GNS_MAX_NT) * GNS_MAX_V * cluster;
}

cudaError_t gns_reg_max_clusters(int64_t seg_len, int64_t S, bool bf16, int cluster, int *clusters)
{
    *clusters = 0;
    if (cluster < 1 || cluster > GNS_MAX_CLUSTER || (cluster & (cluster - 1)) != 0)
        return cudaErrorInvalidValue;
    int nt = 0, idx = 0, dev = 0;
    const RegKernel k = reg_kernel(seg_len, S, bf16, cluster, &nt, &idx);
    if (!k)
        return cudaErrorInvalidValue;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::call_once(g_active_init, [] {
        for (auto &a : g_active)
            for (auto &b : a)
                for (auto &c : b)
                    for (auto &v : c)
                        v.store(-1);
    });
    std::atomic<int> *slot =
        dev >= 0 && dev < GNS_DEVICES ? &g_active[dev][bf16 ? 1 : 0][idx][log2_cluster(cluster)] : nullptr;
    if (slot) {
        const int known = slot->load();
        if (known >= 0) {
            *clusters = known;
            return cudaSuccess;
        }
    }
    e = query_active(k, nt, cluster, clusters);
    if (e == cudaSuccess && slot)
        slot->store(*clusters);
    return e;
}

cudaError_t gns_reg_launch(const GnSegParams &p, bool bf16, int cluster, cudaStream_t stream)
{
    int nt = 0, idx = 0;
    const RegKernel k = reg_kernel(p.seg_len, p.S, bf16, cluster, &nt, &idx);
    if (!k)
        return cudaErrorInvalidValue;
    int active = 0;
    cudaError_t e = gns_reg_max_clusters(p.seg_len, p.S, bf16, cluster, &active);
    if (e != cudaSuccess)
        return e;
    if (active < 1)
        return cudaErrorInvalidConfiguration;
    // every co-resident cluster walks segments; no more clusters than segments
    int64_t clusters = active;
    if (clusters > p.rows)
        clusters = p.rows;
    GnSegParams args = p;
    args.parts = cluster;
    const unsigned grid = static_cast<unsigned>(clusters * cluster);
    if (cluster == 1) {
        k<<<grid, nt, 0, stream>>>(args);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr;
    cluster_config(&cfg, &attr, nt, cluster, grid, stream);
    return cudaLaunchKernelEx(&cfg, k, args);
}

namespace {

// Streamed variants: GroupNorm (act) in 128-thread CTAs, LayerNorm rows in
// 256-thread CTAs, with the same slices (1,024, 2,048 or, bf16, 4,096
// vectors a CTA).  Measured on GB300, each build timed alone (us, 256 -> 128
// threads): GN NCHW (8,512,64,64) fp32 27.0 -> 26.7, bf16 20.7 -> 20.5,
// (16,64,128,128)/8 28.6 -> 26.8, (16,512,32,64) bf16 22.6 -> 20.6; LayerNorm
// rows slower with 128 ((256, 65536) 30.8 -> 33.5, bf16 (512, 32768) 22.6 ->
// 26.9).
constexpr int stream_nt(bool act)
{
    return act ? 128 : 256;
}

// Vectors a CTA slice of the streamed kernel holds: bf16 keeps its values
// packed, so twice as many.
constexpr int stream_cap(bool bf16)
{
    return bf16 ? 4096 : 2048;
}

// CTAs per SM a form's registers are sized for.  The 128-thread forms with
// slices of 1,024 vectors (32 registers a thread of fp32, 16 of bf16) are
// sized for 5 (at most 102 registers, none spilled).  bf16 slices of 2,048
// vectors (32 registers) have two forms: 5 CTAs an SM where a group is split
// over twice the CTAs that hold it ("wide": more clusters resident, more
// groups streamed by each), 4 otherwise.  Measured back to back (µs, 4 ->
// 5 CTAs an SM): (64,512,16,16) fp32 13.9 -> 13.1 and bf16 10.9 -> 10.6;
// (8,512,64,64) bf16 split over 8 CTAs 19.6 -> 17.4; (32,512,16,32) bf16,
// one CTA a group, 10.2 -> 11.8, which keeps the 4-CTA form.
template <typename T, int MODE, bool ACT>
RegKernel stream_kernel_for(int per, bool wide, int *idx)
{
    constexpr int NT = stream_nt(ACT);
    constexpr int SMALL = NT == 128 ? 5 : GNS_MIN_CTAS;
    if (per <= 1024) {
        *idx = 0;
        return gns_stream_kernel<T, NT, 1024 / NT, MODE, ACT, SMALL>;
    }
    if (per <= 2048) {
        if constexpr (sizeof(T) == 2 && NT == 128) {
            if (wide) {
                *idx = 3;
                return gns_stream_kernel<T, NT, 2048 / NT, MODE, ACT, 5>;
            }
        }
        *idx = 1;
        return gns_stream_kernel<T, NT, 2048 / NT, MODE, ACT, GNS_MIN_CTAS>;
    }
    if constexpr (sizeof(T) == 2) {
        if (per <= 4096) {
            *idx = 2;
            return gns_stream_kernel<T, NT, 4096 / NT, MODE, ACT, GNS_MIN_CTAS>;
        }
    }
    *idx = -1;
    return nullptr;
}

// Largest slice (vectors) of the form with index idx.
constexpr int stream_shape_per(int idx)
{
    return idx == 3 ? 2048 : 1024 << idx;
}

// GroupNorm (act: LeakyReLU x2) in all three channel maps; LayerNorm (no
// act) is one group of the whole row with per-element gamma/beta (S = 1).
template <typename T>
RegKernel stream_kernel_t(int per, int mode, bool act, bool wide, int *idx)
{
    if (!act)
        return mode == AFF_ROW ? stream_kernel_for<T, AFF_ROW, false>(per, false, idx) : nullptr;
    switch (mode) {
    case AFF_ROW: return stream_kernel_for<T, AFF_ROW, true>(per, wide, idx);
    case AFF_CHAN: return stream_kernel_for<T, AFF_CHAN, true>(per, wide, idx);
    default: return stream_kernel_for<T, AFF_ANY, true>(per, wide, idx);
    }
}

constexpr int GNS_STREAM_SHAPES = 4;                           // forms by slice (stream_kernel_for)
constexpr int GNS_STREAM_VARIANTS = GNS_STREAM_SHAPES * 4;     // x (3 GroupNorm channel maps + LayerNorm)
std::atomic<int> g_stream_active[GNS_DEVICES][2][GNS_STREAM_VARIANTS][5];
std::once_flag g_stream_init;

// Vectors per CTA slice of the streamed kernel: ceil(L4 / cluster), even so
// that bf16 slices start on 16-byte boundaries.
int64_t stream_per(int64_t seg_len, int cluster)
{
    const int64_t L4 = seg_len / 4;
    const int64_t per = (L4 + cluster - 1) / cluster;
    return (per + 1) & ~int64_t(1);
}

size_t stream_smem(int64_t per, bool bf16)
{
    return static_cast<size_t>(GNS_NBUF) * static_cast<size_t>(per) * 4u * (bf16 ? 2u : 4u);
}

} // namespace

cudaError_t gns_stream_max_clusters(int64_t seg_len, int64_t S, bool bf16, bool act, int cluster, bool wide,
                                    int *clusters)
{
    *clusters = 0;
    if (cluster < 1 || cluster > GNS_MAX_CLUSTER || (cluster & (cluster - 1)) != 0)
        return cudaErrorInvalidValue;
    const int64_t per = stream_per(seg_len, cluster);
    if (per > stream_cap(bf16))
        return cudaErrorInvalidValue;
    int idx = 0, dev = 0;
    const int mode = affine_mode(S);
    const RegKernel k = bf16 ? stream_kernel_t<__nv_bfloat16>(static_cast<int>(per), mode, act, wide, &idx)
                             : stream_kernel_t<float>(static_cast<int>(per), mode, act, wide, &idx);
    if (!k)
        return cudaErrorInvalidValue;
    const int shape = idx;
    idx += GNS_STREAM_SHAPES * (act ? mode : 3);
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::call_once(g_stream_init, [] {
        for (auto &a : g_stream_active)
            for (auto &b : a)
                for (auto &c : b)
                    for (auto &v : c)
                        v.store(-1);
    });
    // occupancy depends on the dynamic shared memory, i.e. on per: cache only
    // the full-slice case (per of 1024, 2048 or 4096), query the others
    const size_t smem = stream_smem(per, bf16);
    const int shape_per = stream_shape_per(shape);
    const bool cacheable = per == shape_per;
    std::atomic<int> *slot = cacheable && dev >= 0 && dev < GNS_DEVICES
                                 ? &g_stream_active[dev][bf16 ? 1 : 0][idx][log2_cluster(cluster)]
                                 : nullptr;
    if (slot) {
        const int known = slot->load();
        if (known >= 0) {
            *clusters = known;
            return cudaSuccess;
        }
    }
    // the attribute covers the variant's largest slice, so any launch of it fits
    const size_t smem_max = stream_smem(shape_per, bf16);
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_max));
    if (e == cudaSuccess && cluster > 8)
        e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess)
        return e;
    const int nt = stream_nt(act);
    if (cluster == 1) {
        int per_sm = 0, sms = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, nt, smem);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        *clusters = per_sm * sms;
    } else {
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr;
        cluster_config(&cfg, &attr, nt, cluster, static_cast<unsigned>(cluster), 0);
        cfg.dynamicSmemBytes = smem;
        e = cudaOccupancyMaxActiveClusters(clusters, k, &cfg);
    }
    if (e == cudaSuccess && slot)
        slot->store(*clusters);
    return e;
}

int64_t gns_stream_capacity4(bool bf16)
{
    return stream_cap(bf16);
}

cudaError_t gns_stream_launch(const GnSegParams &p, bool bf16, bool act, int cluster, bool wide, cudaStream_t stream)
{
    int active = 0;
    cudaError_t e = gns_stream_max_clusters(p.seg_len, p.S, bf16, act, cluster, wide, &active);
    if (e != cudaSuccess)
        return e;
    if (active < 1)
        return cudaErrorInvalidConfiguration;
    const int64_t per = stream_per(p.seg_len, cluster);
    int idx = 0;
    const int mode = affine_mode(p.S);
    const RegKernel k = bf16 ? stream_kernel_t<__nv_bfloat16>(static_cast<int>(per), mode, act, wide, &idx)
                             : stream_kernel_t<float>(static_cast<int>(per), mode, act, wide, &idx);
    int64_t clusters = active;
    if (clusters > p.rows)
        clusters = p.rows;
    GnSegParams args = p;
    args.parts = cluster;
    args.per4 = static_cast<int>(per);
    const size_t smem = stream_smem(per, bf16);
    // The GroupNorm form is launched with programmatic stream serialization:
    // each CTA lets the next kernel be scheduled once its last segment's
    // statistics are merged, so the next call's launch overlaps this one's
    // last writes (back to back, µs per call: (8,512,64,64) bf16 20.4 ->
    // 17.9, fp32 26.7 -> 26.3; (64,512,16,16) fp32 16.4 -> 13.8).  Letting it
    // be scheduled at the start measured slower (fp32 (8,512,64,64) 29.5-29.8
    // us: the next grid's clusters took SMs while this one still ran), and
    // LayerNorm rows measured slower with either trigger ((256, 65536) fp32
    // 30.8 -> 33.2 us, (512, 32768) bf16 22.6 -> 25.2 us), so they launch
    // plainly and the kernel's wait and trigger do nothing.
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    cluster_config(&cfg, &attr[0], stream_nt(act), cluster, static_cast<unsigned>(clusters * cluster), stream);
    cfg.dynamicSmemBytes = smem;
    if (cluster == 1)
        cfg.numAttrs = 0;
    if (act) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        ++cfg.numAttrs;
    }
    return cudaLaunchKernelEx(&cfg, k, args);
}

cudaError_t gns_split_apply_launch(const GnSegParams &p, bool bf16, bool vec4, cudaStream_t stream)
{
    dim3 grid(static_cast<unsigned>(p.parts), static_cast<unsigned>(p.rows < 65535 ? p.rows : 65535));
    if (bf16)
        return vec4 ? launch_pdl(gns_split_apply_kernel<__nv_bfloat16, true>, grid, dim3(GS_T), 0, stream, p)
                    : launch_pdl(gns_split_apply_kernel<__nv_bfloat16, false>, grid, dim3(GS_T), 0, stream, p);
    return vec4 ? launch_pdl(gns_split_apply_kernel<float, true>, grid, dim3(GS_T), 0, stream, p)
                : launch_pdl(gns_split_apply_kernel<float, false>, grid, dim3(GS_T), 0, stream, p);
}

int64_t gns_team_max_items()
{
    return int64_t(32) * TEAM_W;
}

// CTAs of one team kernel resident per SM (team_threads<E>() threads, no
// dynamic shared memory), looked up once per kernel; 0 if the lookup fails.
template <typename T, int E, int MODE, int WMAX>
int team_resident()
{
    static const int n = [] {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, gns_team_kernel<T, E, MODE, WMAX>, team_threads<E>(), 0) !=
            cudaSuccess) {
            cudaGetLastError();
            b = 0;
        }
        return b;
    }();
    return n;
}

// Grid: 4-element items take a persistent grid, exactly the CTAs resident at
// once (each CTA walks its segments with the next one's loads in flight);
// measured faster than 8 CTAs per SM (groups of 48 channels, fp32: 21.8 vs
// 23.8 us; bf16 20.1 vs 20.9 us), while one CTA more per SM than resident
// was the slowest.  2- and 1-element items keep 8 CTAs per SM (a persistent
// grid was slower for them: groups of 30, fp32, 64 vs 40 us).
template <typename T, int E, int MODE, int WMAX>
cudaError_t team_launch_k(const GnSegParams &p, int64_t blocks, int sm_count, int tlog, int W, cudaStream_t stream)
{
    int per_sm = 8;
    if (E == 4) {
        const int r = team_resident<T, E, MODE, WMAX>();
        if (r > 0)
            per_sm = r;
    }
    const int64_t cap = static_cast<int64_t>(sm_count) * per_sm;
    if (blocks > cap)
        blocks = cap;
    return launch_pdl(gns_team_kernel<T, E, MODE, WMAX>, dim3(static_cast<unsigned>(blocks)), dim3(team_threads<E>()),
                      0, stream, p, tlog, W);
}

template <typename T, int WMAX>
cudaError_t team_launch_w(const GnSegParams &p, int elems, int64_t blocks, int sm_count, int tlog, int W,
                          cudaStream_t stream)
{
    const int mode = affine_mode(p.S);
    if (elems == 4) {
        switch (mode) {
        case AFF_ROW: return team_launch_k<T, 4, AFF_ROW, WMAX>(p, blocks, sm_count, tlog, W, stream);
        case AFF_CHAN: return team_launch_k<T, 4, AFF_CHAN, WMAX>(p, blocks, sm_count, tlog, W, stream);
        default: return team_launch_k<T, 4, AFF_ANY, WMAX>(p, blocks, sm_count, tlog, W, stream);
        }
    }
    if (elems == 2)
        return mode == AFF_ROW ? team_launch_k<T, 2, AFF_ROW, WMAX>(p, blocks, sm_count, tlog, W, stream)
                               : team_launch_k<T, 2, AFF_ANY, WMAX>(p, blocks, sm_count, tlog, W, stream);
    return mode == AFF_ROW ? team_launch_k<T, 1, AFF_ROW, WMAX>(p, blocks, sm_count, tlog, W, stream)
                           : team_launch_k<T, 1, AFF_ANY, WMAX>(p, blocks, sm_count, tlog, W, stream);
}

template <typename T>
cudaError_t team_launch_t(const GnSegParams &p, int elems, int sm_count, cudaStream_t stream)
{
    if ((elems != 1 && elems != 2 && elems != 4) || p.seg_len % elems != 0)
        return cudaErrorInvalidValue;
    const int64_t items = p.seg_len / elems;
    if (items < 1 || items > gns_team_max_items())
        return cudaErrorInvalidValue;
    // the narrowest team that gives each lane at most TEAM_TARGET_W items,
    // up to a warp (at most TEAM_W items a lane)
    int tlog = 0;
    while (tlog < 5 && (int64_t(1) << tlog) * TEAM_TARGET_W < items)
        ++tlog;
    const int Tn = 1 << tlog;
    const int W = static_cast<int>((items + Tn - 1) / Tn);
    const int64_t teams_per_cta = (elems == 4 ? team_threads<4>() : team_threads<1>()) / Tn;
    const int64_t blocks = (p.rows + teams_per_cta - 1) / teams_per_cta;
    if (W <= 2)
        return team_launch_w<T, 2>(p, elems, blocks, sm_count, tlog, W, stream);
    if (W <= 4)
        return team_launch_w<T, 4>(p, elems, blocks, sm_count, tlog, W, stream);
    return team_launch_w<T, TEAM_W>(p, elems, blocks, sm_count, tlog, W, stream);
}

cudaError_t gns_team_launch(const GnSegParams &p, bool bf16, int elems, int sm_count, cudaStream_t stream)
{
    return bf16 ? team_launch_t<__nv_bfloat16>(p, elems, sm_count, stream)
                : team_launch_t<float>(p, elems, sm_count, stream);
}

cudaError_t gns_warp_launch(const GnSegParams &p, bool bf16, int sm_count, cudaStream_t stream)
{
    int64_t blocks = (p.rows + 7) / 8;
    const int64_t cap = static_cast<int64_t>(sm_count) * 16;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    if (bf16)
        gns_warp_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    else
        gns_warp_kernel<float><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

} // namespace normk
