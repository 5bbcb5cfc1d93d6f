// gn_kernels.cu - GroupNorm over contiguous channel groups of each row, fused
// with LeakyReLU and x + x (GroupNorm page, POPCORNBENCH transcript
// "Kimi-K2.6 l2_p62": groups of M = C/G contiguous channels, population
// variance, per-channel affine, LeakyReLU(t) = max(0,t) + slope*min(0,t),
// then x + x).
//
// Vector path: one thread owns 4 consecutive channels (a 4-element vector:
// 16 bytes of fp32 or 8 of bf16), so a group of M channels is TPG = M/4
// adjacent lanes and a warp covers 128 contiguous elements.  Mean and then
// the exact M2 about the mean are reduced over the TPG lanes with xor
// shuffles (the group's values never leave registers), the epilogue is
// applied in fp32 registers and the vector is stored once.  A CTA keeps its
// columns' gamma/beta in registers and walks rows with two rows of x loads in
// flight, held as loaded (bf16 packed, two registers a vector) until their
// turn.  Every byte of x is read once and every byte of y written once.
//
// bf16 groups of 8 or more channels with 16-byte aligned tensors take a
// wider form: a thread owns 8 channels (one 16-byte load, four registers
// held packed) and keeps three rows of loads in flight, so an SM has about
// as many bytes of x in flight as in fp32 at half the bytes per element.
#include "norm_internal.cuh"

namespace normk {

namespace {

constexpr int GN_THREADS = 256;  // the 8-channel bf16 form
// The 4-channel form: 128-thread CTAs.  Measured at (1024, 8192) fp32, back
// to back: 11.84-11.90 us with grids of 16 to 32 CTAs of 128 an SM, against
// 12.14-12.16 us with 256-thread CTAs (8 an SM) and 12.28 us with 512.
constexpr int GN4_THREADS = 128;

template <int TPG>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = TPG / 2; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// A prefetched 4-element vector as loaded: fp32 as a float4, bf16 packed
// (two registers), widened when its row's turn comes.
template <typename T>
struct Raw4;

template <>
struct Raw4<float> {
    using type = float4;
    static __device__ __forceinline__ type load(const float *p, uint64_t pol) { return Io<float>::ld4_stream(p, pol); }
    static __device__ __forceinline__ type zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    static __device__ __forceinline__ float4 get(const type &r) { return r; }
};

template <>
struct Raw4<__nv_bfloat16> {
    using type = uint2;
    static __device__ __forceinline__ type load(const __nv_bfloat16 *p, uint64_t pol)
    {
        uint2 r;
        asm("ld.global.L1::no_allocate.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
            : "=r"(r.x), "=r"(r.y)
            : "l"(p), "l"(pol));
        return r;
    }
    static __device__ __forceinline__ type zero() { return make_uint2(0u, 0u); }
    static __device__ __forceinline__ float4 get(const type &r) { return Io<__nv_bfloat16>::unpack(r.x, r.y); }
};

// grid: x = column blocks of GN4_THREADS*U vectors, y = row walkers.
// x, y: [N][C] of T; "vector" = 4 consecutive channels; C4 = C / 4.
// A CTA owns a fixed block of GN4_THREADS * U vectors of columns and walks
// rows n = blockIdx.y, + gridDim.y, ...: gamma/beta of its columns are
// loaded once, and the next two rows' x are loaded while the current row is
// reduced and written, so every thread keeps two rows of loads in flight.
template <typename T, int TPG, int U>
__global__ void __launch_bounds__(GN4_THREADS) gn_vec4_kernel(const T *x, const T *__restrict__ gamma,
                                                             const T *__restrict__ beta, T *y,
                                                             int64_t N, int C4, float invM, float eps,
                                                             float slope)
{
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    pdl_begin();
    const int col0 = blockIdx.x * (GN4_THREADS * U) + threadIdx.x;
    using R = Raw4<T>;
    float2 g[U][2], b[U][2]; // gamma/beta of the vector's two pairs
    typename R::type cur[U], nxt[U], nx2[U];
    // gamma and beta are held doubled: 2 LReLU(t) = LReLU(2 t) and doubling is
    // exact, so the x + x costs nothing per element and the result is the same
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int c = col0 + u * GN4_THREADS;
        const bool in = c < C4;
        const float4 gv = (in && gamma) ? Io<T>::ld4_ro(gamma + 4 * c, pol_keep) : make_float4(1.f, 1.f, 1.f, 1.f);
        const float4 bv = (in && beta) ? Io<T>::ld4_ro(beta + 4 * c, pol_keep) : make_float4(0.f, 0.f, 0.f, 0.f);
        g[u][0] = make_float2(gv.x + gv.x, gv.y + gv.y);
        g[u][1] = make_float2(gv.z + gv.z, gv.w + gv.w);
        b[u][0] = make_float2(bv.x + bv.x, bv.y + bv.y);
        b[u][1] = make_float2(bv.z + bv.z, bv.w + bv.w);
    }
    const float2 slope2 = make_float2(slope, slope);
    // LReLU(t) = max(t, slope t) for slope <= 1, min(t, slope t) above
    const bool steep = slope > 1.f;
    auto load_row = [&](int64_t n, typename R::type *dst) {
        const T *xr = x + n * C4 * 4;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = col0 + u * GN4_THREADS;
            dst[u] = c < C4 ? R::load(xr + 4 * c, pol_stream) : R::zero();
        }
    };
    if (blockIdx.y < N)
        load_row(blockIdx.y, nxt);
    if (blockIdx.y + gridDim.y < N)
        load_row(blockIdx.y + gridDim.y, nx2);
    for (int64_t n = blockIdx.y; n < N; n += gridDim.y) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            cur[u] = nxt[u];
            nxt[u] = nx2[u];
        }
        // with y == x the rows ahead are other rows: loading them now
        // cannot race with this row's stores
        if (n + 2 * gridDim.y < N)
            load_row(n + 2 * gridDim.y, nx2);
        T *yr = y + n * C4 * 4;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = col0 + u * GN4_THREADS;
            // C4 is a multiple of TPG, so whole groups are in or out of range
            // together and every lane takes part in the shuffles.  The
            // arithmetic is in f32x2 pairs.
            const float4 cv = R::get(cur[u]);
            const float2 xl = make_float2(cv.x, cv.y), xh = make_float2(cv.z, cv.w);
            const float2 s2 = __fadd2_rn(xl, xh);
            const float mean = group_sum<TPG>(s2.x + s2.y) * invM;
            const float2 nm = make_float2(-mean, -mean);
            const float2 dl = __fadd2_rn(xl, nm), dh = __fadd2_rn(xh, nm);
            const float2 q2 = __ffma2_rn(dh, dh, __fmul2_rn(dl, dl));
            const float m2 = group_sum<TPG>(q2.x + q2.y);
            const float rstd = rsqrtf(fmaf(m2, invM, eps));
            if (c < C4) {
                const float2 r2 = make_float2(rstd, rstd);
                float2 tl = __ffma2_rn(__fmul2_rn(dl, r2), g[u][0], b[u][0]);
                float2 th = __ffma2_rn(__fmul2_rn(dh, r2), g[u][1], b[u][1]);
                const float2 ul = __fmul2_rn(tl, slope2), uh = __fmul2_rn(th, slope2);
                tl = steep ? make_float2(fminf(tl.x, ul.x), fminf(tl.y, ul.y))
                           : make_float2(fmaxf(tl.x, ul.x), fmaxf(tl.y, ul.y));
                th = steep ? make_float2(fminf(th.x, uh.x), fminf(th.y, uh.y))
                           : make_float2(fmaxf(th.x, uh.x), fmaxf(th.y, uh.y));
                Io<T>::st4_stream(yr + 4 * c, make_float4(tl.x, tl.y, th.x, th.y), pol_stream);
            }
        }
    }
}


// bf16 vector path with 8 channels (one 16-byte access) a thread: a group of
// M channels is TPG = M/8 adjacent lanes, and a warp covers 256 contiguous
// elements (512 bytes).  Each row's x is held as loaded (four registers) from
// its load, GN8_AHEAD rows ahead of the row being reduced, until its turn.
constexpr int GN8_AHEAD = 3;
// One resident wave of 5 CTAs of 256 threads an SM (the launch bound holds
// the kernel to 48 registers), so a row walker takes at most 6 rows of 1,024.
// Measured at (1024, 8192) bf16, back to back: 7.73 us, against 7.95 us with
// 4 CTAs an SM and four rows ahead (53 registers, at most 7 rows a walker)
// and 8.97 us for the 4-channel form; 5 CTAs with four rows ahead spilled
// and took 8.13 us, 6 CTAs with three rows ahead 7.90 us; 2, 5, 6 and 8 rows
// ahead, two vectors a thread and 6 or 8 CTAs at four rows ahead 8.15-9.8 us.
constexpr int GN8_CTAS_PER_SM = 5;

__device__ __forceinline__ float2 bf16_pair(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ uint4 ld16_stream(const void *p, uint64_t pol)
{
    uint4 r;
    asm("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p), "l"(pol));
    return r;
}

__device__ __forceinline__ uint4 ld16_ro(const void *p, uint64_t pol)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p), "l"(pol));
    return r;
}

__device__ __forceinline__ void st16_stream(void *p, uint4 v, uint64_t pol)
{
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

// grid: x = column blocks of GN_THREADS vectors of 8, y = row walkers.
// x, y: [N][C] of bf16; C8 = C / 8.  Same walk as gn_vec4_kernel.
template <int TPG>
__global__ void __launch_bounds__(GN_THREADS, GN8_CTAS_PER_SM) gn_vec8_bf16_kernel(const __nv_bfloat16 *x,
                                                                  const __nv_bfloat16 *__restrict__ gamma,
                                                                  const __nv_bfloat16 *__restrict__ beta,
                                                                  __nv_bfloat16 *y, int64_t N, int C8, float invM,
                                                                  float eps, float slope)
{
    constexpr int D = GN8_AHEAD;
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    pdl_begin();
    const int c = blockIdx.x * GN_THREADS + threadIdx.x;
    const bool in = c < C8;
    // doubled gamma/beta of the vector's four pairs (see gn_vec4_kernel)
    float2 g[4], b[4];
    {
        constexpr uint32_t one2 = 0x3f803f80u; // two bf16 1.0
        const uint4 gv = (in && gamma) ? ld16_ro(gamma + 8 * c, pol_keep) : make_uint4(one2, one2, one2, one2);
        const uint4 bv = (in && beta) ? ld16_ro(beta + 8 * c, pol_keep) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 gp = bf16_pair(gw[j]), bp = bf16_pair(bw[j]);
            g[j] = make_float2(gp.x + gp.x, gp.y + gp.y);
            b[j] = make_float2(bp.x + bp.x, bp.y + bp.y);
        }
    }
    const float2 slope2 = make_float2(slope, slope);
    const bool steep = slope > 1.f;
    uint4 buf[D + 1]; // buf[0]: the row being reduced; buf[k]: k rows ahead
    auto load_row = [&](int64_t n) {
        return in ? ld16_stream(x + (n * C8 + c) * 8, pol_stream) : make_uint4(0u, 0u, 0u, 0u);
    };
#pragma unroll
    for (int k = 0; k < D; ++k)
        if (blockIdx.y + int64_t(k) * gridDim.y < N)
            buf[k + 1] = load_row(blockIdx.y + int64_t(k) * gridDim.y);
    for (int64_t n = blockIdx.y; n < N; n += gridDim.y) {
#pragma unroll
        for (int k = 0; k < D; ++k)
            buf[k] = buf[k + 1];
        // with y == x the rows ahead are other rows: loading them now cannot
        // race with this row's stores
        if (n + int64_t(D) * gridDim.y < N)
            buf[D] = load_row(n + int64_t(D) * gridDim.y);
        // C8 is a multiple of TPG, so whole groups are in or out of range
        // together and every lane takes part in the shuffles
        float2 p[4] = {bf16_pair(buf[0].x), bf16_pair(buf[0].y), bf16_pair(buf[0].z), bf16_pair(buf[0].w)};
        const float2 s2 = __fadd2_rn(__fadd2_rn(p[0], p[1]), __fadd2_rn(p[2], p[3]));
        const float mean = group_sum<TPG>(s2.x + s2.y) * invM;
        const float2 nm = make_float2(-mean, -mean);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            p[j] = __fadd2_rn(p[j], nm);
        float2 q2 = __fmul2_rn(p[0], p[0]);
#pragma unroll
        for (int j = 1; j < 4; ++j)
            q2 = __ffma2_rn(p[j], p[j], q2);
        const float m2 = group_sum<TPG>(q2.x + q2.y);
        const float rstd = rsqrtf(fmaf(m2, invM, eps));
        if (in) {
            const float2 r2 = make_float2(rstd, rstd);
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float2 t = __ffma2_rn(__fmul2_rn(p[j], r2), g[j], b[j]);
                const float2 w = __fmul2_rn(t, slope2);
                t = steep ? make_float2(fminf(t.x, w.x), fminf(t.y, w.y))
                          : make_float2(fmaxf(t.x, w.x), fmaxf(t.y, w.y));
                o[j] = pack_bf16x2(t.x, t.y);
            }
            st16_stream(y + (n * C8 + c) * 8, make_uint4(o[0], o[1], o[2], o[3]), pol_stream);
        }
    }
}

template <int TPG>
cudaError_t launch_vec8(const void *x, const void *gamma, const void *beta, void *y, int64_t N, int64_t C,
                        int64_t M, float eps, float slope, int sm_count, cudaStream_t stream)
{
    const int C8 = static_cast<int>(C / 8);
    const int gx = (C8 + GN_THREADS - 1) / GN_THREADS;
    int64_t gy = (static_cast<int64_t>(sm_count) * GN8_CTAS_PER_SM + gx - 1) / gx;
    if (gy > N)
        gy = N;
    if (gy > 65535)
        gy = 65535;
    if (gy < 1)
        gy = 1;
    dim3 grid(gx, static_cast<unsigned>(gy));
    return launch_pdl(gn_vec8_bf16_kernel<TPG>, grid, dim3(GN_THREADS), 0, stream,
                      static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(gamma),
                      static_cast<const __nv_bfloat16 *>(beta), static_cast<__nv_bfloat16 *>(y), N, C8,
                      1.0f / static_cast<float>(M), eps, slope);
}


template <typename T, int TPG, int U>
cudaError_t launch_vec(const void *x, const void *gamma, const void *beta, void *y, int64_t N, int64_t C,
                       int64_t M, float eps, float slope, int sm_count, cudaStream_t stream)
{
    const int C4 = static_cast<int>(C / 4);
    const int per_block = GN4_THREADS * U;
    const int gx = (C4 + per_block - 1) / per_block;
    // Grid sized for 20 CTAs of 128 threads per SM; each walks N / gy rows.
    // About 9 are resident at once (54 registers a thread), so the launch
    // runs as two waves: with 256-thread CTAs two waves also measured faster
    // than one (fp32 12.2 vs 12.4 us, bf16 9.0 vs 10.0 us a call back to
    // back); with 128 threads, 16 to 32 an SM measured the same (11.84-11.90
    // us) and 12 slower (12.41 us).
    constexpr int CTAS_PER_SM = 20;
    int64_t gy = (static_cast<int64_t>(sm_count) * CTAS_PER_SM + gx - 1) / gx;
    if (gy > N)
        gy = N;
    if (gy > 65535)
        gy = 65535;
    if (gy < 1)
        gy = 1;
    dim3 grid(gx, static_cast<unsigned>(gy));
    return launch_pdl(gn_vec4_kernel<T, TPG, U>, grid, dim3(GN4_THREADS), 0, stream, static_cast<const T *>(x),
                      static_cast<const T *>(gamma), static_cast<const T *>(beta), static_cast<T *>(y), N, C4,
                      1.0f / static_cast<float>(M), eps, slope);
}

} // namespace

// Two vectors a thread per row.
template <typename T>
cudaError_t gn_vec4_launch_t(const void *x, const void *gamma, const void *beta, void *y, int64_t N, int64_t C,
                             int64_t M, float eps, float slope, int sm_count, cudaStream_t stream)
{
    constexpr int U = 2;
    switch (M) {
    case 4: return launch_vec<T, 1, U>(x, gamma, beta, y, N, C, M, eps, slope, sm_count, stream);
    case 8: return launch_vec<T, 2, U>(x, gamma, beta, y, N, C, M, eps, slope, sm_count, stream);
    case 16: return launch_vec<T, 4, U>(x, gamma, beta, y, N, C, M, eps, slope, sm_count, stream);
    case 32: return launch_vec<T, 8, U>(x, gamma, beta, y, N, C, M, eps, slope, sm_count, stream);
    case 64: return launch_vec<T, 16, U>(x, gamma, beta, y, N, C, M, eps, slope, sm_count, stream);
    case 128: return launch_vec<T, 32, U>(x, gamma, beta, y, N, C, M, eps, slope, sm_count, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t gn_vec4_launch(const void *x, const void *gamma, const void *beta, void *y, int64_t N, int64_t C,
                           int64_t M, float eps, float slope, bool bf16, int sm_count, cudaStream_t stream)
{
    const bool a16 = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) |
                       reinterpret_cast<uintptr_t>(gamma) | reinterpret_cast<uintptr_t>(beta)) & 15) == 0;
    if (bf16 && a16) {
        switch (M) {
        case 8: return launch_vec8<1>(x, gamma, beta, y, N, C, M, eps, slope, sm_count, stream);
        case 16: return launch_vec8<2>(x, gamma, beta, y, N, C, M, eps, slope, sm_count, stream);
        case 32: return launch_vec8<4>(x, gamma, beta, y, N, C, M, eps, slope, sm_count, stream);
        case 64: return launch_vec8<8>(x, gamma, beta, y, N, C, M, eps, slope, sm_count, stream);
        case 128: return launch_vec8<16>(x, gamma, beta, y, N, C, M, eps, slope, sm_count, stream);
        default: break; // groups of 4 channels: the 4-channel form
        }
    }
    return bf16 ? gn_vec4_launch_t<__nv_bfloat16>(x, gamma, beta, y, N, C, M, eps, slope, sm_count, stream)
                : gn_vec4_launch_t<float>(x, gamma, beta, y, N, C, M, eps, slope, sm_count, stream);
}

} // namespace normk
