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
    const int64_t bx = (S + RMS_THREADS - 1) / RMS_THREADS;
    if (bx > 0x7fffffff)
        return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(B < 65535 ? B : 65535));
    const int Ci = static_cast<int>(C);
    const float invC = 1.0f / static_cast<float>(C);
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
