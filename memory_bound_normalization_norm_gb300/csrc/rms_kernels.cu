// rms_kernels.cu - RMSNorm over dim 1 of x[B][C][S] (RMSNorm page,
// POPCORNBENCH transcript "Kimi-K2.6 l1_p36": rms = sqrt(mean_c x^2 + eps),
// y = x / rms; the channel stride is S = H*W elements).
//
// Mapping: thread <-> spatial position s, so for every channel the 32 lanes
// of a warp touch 32 consecutive floats (128 contiguous bytes, whole
// sectors).  The position's C values are loaded into registers (all C loads
// of a thread are independent, so they are all in flight at once), reduced,
// scaled and stored from registers: x is read from HBM exactly once.
// C > 128 falls back to a two-read kernel.
#include "norm_internal.cuh"

namespace normk {

namespace {

constexpr int RMS_THREADS = 128;

// grid: x = position blocks, y = batch entries (folded by gridDim.y).
// EXACT: C == CMAX, so no channel is predicated off.  The channel addresses
// are walked with a running pointer: materializing all CMAX 64-bit addresses
// at once would cost 2*CMAX registers.
// Register cap: exact C <= 64 fits in 128 registers (4 CTAs of 128 threads
// per SM); C = 128 and the predicated (C < CMAX) forms get up to 255.
template <typename T, int CMAX, bool EXACT>
__global__ void __launch_bounds__(RMS_THREADS, (EXACT && CMAX <= 64) ? 4 : 2) rms_reg_kernel(const T *x, T *y, int64_t B, int C,
                                                                 int64_t S, float invC, float eps)
{
    pdl_begin();
    const uint64_t pol = policy_evict_first();
    const int64_t s = static_cast<int64_t>(blockIdx.x) * RMS_THREADS + threadIdx.x;
    if (s >= S)
        return;
    for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
        const T *xp = x + b * C * S + s;
        float v[CMAX];
#pragma unroll
        for (int c = 0; c < CMAX; ++c) {
            v[c] = (EXACT || c < C) ? Io<T>::ld1_stream(xp, pol) : 0.f;
            xp += S;
        }
        // four independent partial sums, combined in a fixed order
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int c = 0; c < CMAX; c += 4) {
            a0 = fmaf(v[c], v[c], a0);
            if (c + 1 < CMAX)
                a1 = fmaf(v[c + 1], v[c + 1], a1);
            if (c + 2 < CMAX)
                a2 = fmaf(v[c + 2], v[c + 2], a2);
            if (c + 3 < CMAX)
                a3 = fmaf(v[c + 3], v[c + 3], a3);
        }
        const float inv = rsqrtf(fmaf((a0 + a1) + (a2 + a3), invC, eps));
        T *yp = y + b * C * S + s;
#pragma unroll
        for (int c = 0; c < CMAX; ++c) {
            if (EXACT || c < C)
                Io<T>::st1_stream(yp, v[c] * inv, pol);
            yp += S;
        }
    }
}

// bf16 with S even and 4-byte aligned tensors: thread <-> two adjacent
// positions, so a warp's load or store of one channel is 32 x 4 = 128
// contiguous bytes (as in fp32) and each thread keeps twice the bytes in
// flight of a one-position thread.  The C bf16 pairs stay packed in
// registers; the sums of squares and the scaling run in f32x2 pairs.
__device__ __forceinline__ uint32_t ld_u32_stream(const void *p, uint64_t pol)
{
    uint32_t v;
    asm("ld.global.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ void st_u32_stream(void *p, uint32_t v, uint64_t pol)
{
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.u32 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(pol) : "memory");
}

// Exact C only (every channel loaded unpredicated): C = 64 takes about 160
// registers (3 CTAs per SM, still 96 KB of loads in flight per SM against
// 64 KB for one position a thread); smaller C fit 4 CTAs per SM.
template <int CMAX>
__global__ void __launch_bounds__(RMS_THREADS, CMAX <= 32 ? 4 : 3)
    rms_bf16x2_kernel(const __nv_bfloat16 *x, __nv_bfloat16 *y, int64_t B, int C, int64_t S, float invC, float eps)
{
    pdl_begin();
    const uint64_t pol = policy_evict_first();
    const int64_t s = 2 * (static_cast<int64_t>(blockIdx.x) * RMS_THREADS + threadIdx.x);
    if (s >= S)
        return;
    for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
        const __nv_bfloat16 *xp = x + b * C * S + s;
        uint32_t v[CMAX];
#pragma unroll
        for (int c = 0; c < CMAX; ++c) {
            v[c] = ld_u32_stream(xp, pol);
            xp += S;
        }
        // four independent pairs of partial sums, combined in a fixed order
        float2 a[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < CMAX; ++c) {
            const float2 t = make_float2(__uint_as_float(v[c] << 16), __uint_as_float(v[c] & 0xffff0000u));
            a[c & 3] = __ffma2_rn(t, t, a[c & 3]);
        }
        const float2 sum = __fadd2_rn(__fadd2_rn(a[0], a[1]), __fadd2_rn(a[2], a[3]));
        const float2 inv = make_float2(rsqrtf(fmaf(sum.x, invC, eps)), rsqrtf(fmaf(sum.y, invC, eps)));
        __nv_bfloat16 *yp = y + b * C * S + s;
#pragma unroll
        for (int c = 0; c < CMAX; ++c) {
            const float2 t = __fmul2_rn(make_float2(__uint_as_float(v[c] << 16), __uint_as_float(v[c] & 0xffff0000u)),
                                        inv);
            st_u32_stream(yp, pack_bf16x2(t.x, t.y), pol);
            yp += S;
        }
    }
}

// Any C: sum of squares in one pass, then a second pass re-reads x to scale.
template <typename T>
__global__ void __launch_bounds__(RMS_THREADS) rms_generic_kernel(const T *x, T *y, int64_t B, int64_t C,
                                                                  int64_t S, float invC, float eps)
{
    const int64_t s = static_cast<int64_t>(blockIdx.x) * RMS_THREADS + threadIdx.x;
    if (s >= S)
        return;
    for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
        const T *xp = x + b * C * S + s;
        T *yp = y + b * C * S + s;
        float a = 0.f;
        for (int64_t c = 0; c < C; ++c) {
            const float v = Io<T>::ld1(xp + c * S);
            a = fmaf(v, v, a);
        }
        const float inv = rsqrtf(fmaf(a, invC, eps));
        for (int64_t c = 0; c < C; ++c)
            Io<T>::st1(yp + c * S, Io<T>::ld1(xp + c * S) * inv);
    }
}

template <typename T, int CMAX>
cudaError_t launch_reg(const T *x, T *y, int64_t B, int64_t C, int64_t S, float eps, cudaStream_t stream)
{
    const int Ci = static_cast<int>(C);
    const float invC = 1.0f / static_cast<float>(C);
    if constexpr (sizeof(T) == 2 && CMAX <= 64) {
        // two positions a thread where every pair is 4-byte aligned and C is exact
        const bool pairs = C == CMAX && (S & 1) == 0 && (reinterpret_cast<uintptr_t>(x) & 3) == 0 &&
                           (reinterpret_cast<uintptr_t>(y) & 3) == 0;
        if (pairs) {
            const int64_t bx2 = (S / 2 + RMS_THREADS - 1) / RMS_THREADS;
            if (bx2 > 0x7fffffff)
                return cudaErrorInvalidValue;
            dim3 g2(static_cast<unsigned>(bx2), static_cast<unsigned>(B < 65535 ? B : 65535));
            return launch_pdl(rms_bf16x2_kernel<CMAX>, g2, dim3(RMS_THREADS), 0, stream, x, y, B, Ci, S, invC, eps);
        }
    }
    const int64_t bx = (S + RMS_THREADS - 1) / RMS_THREADS;
    if (bx > 0x7fffffff)
        return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(B < 65535 ? B : 65535));
    if (C == CMAX)
        return launch_pdl(rms_reg_kernel<T, CMAX, true>, grid, dim3(RMS_THREADS), 0, stream, x, y, B, Ci, S, invC, eps);
    return launch_pdl(rms_reg_kernel<T, CMAX, false>, grid, dim3(RMS_THREADS), 0, stream, x, y, B, Ci, S, invC, eps);
}

} // namespace

template <typename T>
cudaError_t rms_channel_launch_t(const T *x, T *y, int64_t B, int64_t C, int64_t S, float eps, cudaStream_t stream)
{
    if (C <= 4)
        return launch_reg<T, 4>(x, y, B, C, S, eps, stream);
    if (C <= 8)
        return launch_reg<T, 8>(x, y, B, C, S, eps, stream);
    if (C <= 16)
        return launch_reg<T, 16>(x, y, B, C, S, eps, stream);
    if (C <= 32)
        return launch_reg<T, 32>(x, y, B, C, S, eps, stream);
    if (C <= 64)
        return launch_reg<T, 64>(x, y, B, C, S, eps, stream);
    if (C <= 128)
        return launch_reg<T, 128>(x, y, B, C, S, eps, stream);
    const int64_t bx = (S + RMS_THREADS - 1) / RMS_THREADS;
    if (bx > 0x7fffffff)
        return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(B < 65535 ? B : 65535));
    rms_generic_kernel<T><<<grid, RMS_THREADS, 0, stream>>>(x, y, B, C, S, 1.0f / static_cast<float>(C), eps);
    return cudaGetLastError();
}

cudaError_t rms_channel_launch(const void *x, void *y, int64_t B, int64_t C, int64_t S, float eps, bool bf16,
                               cudaStream_t stream)
{
    if (bf16)
        return rms_channel_launch_t(static_cast<const __nv_bfloat16 *>(x), static_cast<__nv_bfloat16 *>(y), B, C, S,
                                    eps, stream);
    return rms_channel_launch_t(static_cast<const float *>(x), static_cast<float *>(y), B, C, S, eps, stream);
}

} // namespace normk
