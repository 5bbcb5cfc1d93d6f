// ln_noalloc.cu - LayerNorm for callers that cannot allocate device memory.
//
// norm_layer_fwd needs a scratch workspace on two of its paths (the
// persistent kernel's grid-barrier header and tagged records, the two-kernel
// path's per-chunk partials).  Some callers cannot provide one: code that
// runs where cudaMalloc is not allowed (inside a custom allocator's own
// callbacks, in a process whose memory pool is fixed up front, or in a
// plugin that receives only input and output pointers from its host).  For
// them, norm_layer_fwd_noalloc keeps that scratch in a fixed-size array that
// is part of this library's device image, so the call itself never
// allocates.
#include <mutex>

#include "norm_internal.cuh"

namespace {

// The scratch of norm_layer_fwd_noalloc.  Every device that loads the library
// holds these NORM_NOALLOC_SCRATCH_BYTES until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NORM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices]; // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device.  In host code
// the name g_noalloc_scratch is only a host-side stand-in, so the address is
// looked up once per device, with that device current.
norm_status_t scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return NORM_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return NORM_ERR_CUDA;
        }
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return NORM_OK;
}

} // namespace

extern "C" norm_status_t norm_layer_fwd_noalloc(const float *x, const float *gamma, const float *beta, float *y,
                                                int64_t rows, int64_t row_len, float eps, cudaStream_t stream)
{
    // The path norm_layer_fwd takes for this call, and the scratch it needs
    // (none on the row and cluster kernels).
    size_t need = 0;
    norm_status_t st = normapi::layer_fwd_workspace_need(x, gamma, beta, y, rows, row_len, eps, 4, &need);
    if (st != NORM_OK)
        return st;
    if (need > NORM_NOALLOC_SCRATCH_BYTES)
        return NORM_ERR_WORKSPACE;
    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != NORM_OK)
        return st;
    // The array keeps whatever the previous call left in it (another shape's
    // partials, or the state of a call that gave up waiting): start from
    // zeros, as from a fresh workspace, over every byte this path uses.
    if (need > 0 && cudaMemsetAsync(scratch, 0, need, stream) != cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
    }
    return norm_layer_fwd(x, gamma, beta, y, rows, row_len, eps, scratch, NORM_NOALLOC_SCRATCH_BYTES, stream);
}
