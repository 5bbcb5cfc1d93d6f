// norm_internal.cuh - device helpers and launcher declarations shared by the
// kernels of libnormgb300 (sm_103a).  Inline PTX only; no library kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "norm.h"

namespace normk {

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// L2 eviction policies (createpolicy, sm_80+).  evict_first for data that is
// touched once (x, y), evict_last for data re-read by every row (gamma, beta).
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Coherent 128-bit / 32-bit global loads that do not allocate in L1, with an
// L2 eviction policy.  (Coherent rather than .nc so that y == x is safe.)
// Pure loads are not `volatile`: the compiler may schedule them freely, which
// is what lets independent loads of an unrolled loop be in flight together.
__device__ __forceinline__ float4 ld_stream_f4(const float4 *p, uint64_t pol)
{
    float4 v;
    asm("ld.global.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ float ld_stream_f1(const float *p, uint64_t pol)
{
    float v;
    asm("ld.global.L1::no_allocate.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(pol));
    return v;
}

// Read-only (non-coherent path) 128-bit load with an L2 policy: for gamma/beta,
// which the kernels never write.
// A parameter vector (gamma/beta) that every row reads again: read-only and
// L1-allocating, so the rows a CTA walks find it in L1.
__device__ __forceinline__ float4 ld_param_f4(const float4 *p)
{
    float4 v;
    asm("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ld_ro_f4(const float4 *p, uint64_t pol)
{
    float4 v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ void st_stream_f4(float4 *p, float4 v, uint64_t pol)
{
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;"
                 :
                 : "l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ float2 ld_stream_f2(const float2 *p, uint64_t pol)
{
    float2 v;
    asm("ld.global.L1::no_allocate.L2::cache_hint.v2.f32 {%0, %1}, [%2], %3;"
        : "=f"(v.x), "=f"(v.y)
        : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ void st_stream_f2(float2 *p, float2 v, uint64_t pol)
{
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;"
                 :
                 : "l"(p), "f"(v.x), "f"(v.y), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void st_stream_f1(float *p, float v, uint64_t pol)
{
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.f32 [%0], %1, %2;"
                 :
                 : "l"(p), "f"(v), "l"(pol)
                 : "memory");
}

// Plain coherent scalar load (never the read-only path).
__device__ __forceinline__ float ld_plain_f1(const float *p)
{
    float v;
    asm("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// 128-bit load served from L2 (never a possibly stale L1 line): for data
// written by other CTAs of the same kernel after a grid-scope acquire.
__device__ __forceinline__ float4 ld_l2_f4(const float4 *p)
{
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

// ---- programmatic dependent launch
// A kernel launched with launch_pdl may start while the previous kernel in
// its stream is still finishing, so back-to-back calls overlap one kernel's
// launch and tail with the next one's (GroupNorm (1024,8192): 14.4 -> 12.0
// us per call).  pdl_begin() first lets the next kernel of the stream be
// scheduled early, then waits until the previous kernel has completed and
// its writes are visible: it must come before the kernel's first global
// memory access.  Without a programmatic predecessor the wait returns at
// once.  Used by the grid-stride kernels (row LayerNorm, (N, C) GroupNorm,
// RMSNorm) and both kernels of the two-kernel paths.  The streamed cluster
// kernel's GroupNorm form waits first and triggers late (pdl_wait, then
// pdl_trigger once its last segment's statistics are merged); the
// persistent LayerNorm kernel launches normally.
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_begin()
{
    pdl_trigger();
    pdl_wait();
}

// ---- mbarrier + bulk copy (TMA engine, non-tensor form)

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of whether phase `parity` of `bar` has completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, giving up after timeout_ns.
// The first look does not suspend the thread (mbarrier.try_wait may, for a
// hardware-defined time), and a limit below one microsecond, finer than
// %globaltimer is guaranteed to resolve, gives up at that first look if the
// phase is not complete: tiny limits make every wait that is not already
// over give up, deterministically.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t timeout_ns)
{
    if (mbar_test_wait(bar, parity))
        return true;
    if (timeout_ns < 1000)
        return false;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > timeout_ns)
            return false;
    }
    return true;
}

// Bulk copy global -> this CTA's shared memory; completion is signalled on
// `bar` as transaction bytes.  dst, src and bytes must be 16-byte multiples.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// Bulk copy this CTA's shared memory -> global, tracked by the issuing
// thread's bulk async-groups (bulk_commit / bulk_wait_*).  dst, src and
// bytes must be 16-byte multiples.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk group of this thread has finished reading
// its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---- gpu-scope synchronization primitives

// 64-bit load from L2 (bypassing L1) that the compiler may not merge or drop,
// and that the hardware may overlap with other loads (unlike ld.relaxed.gpu,
// whose loads were measured to complete one after another).  A naturally
// aligned 8-byte word written by one 64-bit store is read whole.
__device__ __forceinline__ unsigned long long ld_cg_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.global.cg.b64 %0, [%1];" : "=l"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ unsigned ld_relaxed_gpu_u32(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu_u32(unsigned *p, unsigned v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Record the first device-side failure in the per-device error word.
__device__ __forceinline__ void record_error(unsigned *err, unsigned code)
{
    if (err)
        atomicCAS(err, 0u, code);
}

// Named CTA barrier (ids 1..15; id 0 is __syncthreads) over `count`
// threads, a multiple of 32.
__device__ __forceinline__ void bar_sync_named(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------- element types
// Io<T> moves elements of type T (float, or __nv_bfloat16 with fp32
// arithmetic) between memory and fp32 registers.  The 4-element forms need
// p aligned to 4 elements (16 bytes for fp32, 8 for bf16), the 2-element
// forms to 2 elements.  bf16 -> fp32 is
// exact; fp32 -> bf16 rounds to nearest even (CUDA's __float2bfloat16_rn).
template <typename T>
struct Io;

template <>
struct Io<float> {
    static __device__ __forceinline__ float4 ld4_stream(const float *p, uint64_t pol)
    {
        return ld_stream_f4(reinterpret_cast<const float4 *>(p), pol);
    }
    static __device__ __forceinline__ float4 ld4_ro(const float *p, uint64_t pol)
    {
        return ld_ro_f4(reinterpret_cast<const float4 *>(p), pol);
    }
    static __device__ __forceinline__ float4 ld4_param(const float *p)
    {
        return ld_param_f4(reinterpret_cast<const float4 *>(p));
    }
    static __device__ __forceinline__ void st4_stream(float *p, float4 v, uint64_t pol)
    {
        st_stream_f4(reinterpret_cast<float4 *>(p), v, pol);
    }
    static __device__ __forceinline__ float2 ld2_stream(const float *p, uint64_t pol)
    {
        return ld_stream_f2(reinterpret_cast<const float2 *>(p), pol);
    }
    static __device__ __forceinline__ void st2_stream(float *p, float2 v, uint64_t pol)
    {
        st_stream_f2(reinterpret_cast<float2 *>(p), v, pol);
    }
    static __device__ __forceinline__ float ld1(const float *p) { return ld_plain_f1(p); }
    static __device__ __forceinline__ float ld1_stream(const float *p, uint64_t pol) { return ld_stream_f1(p, pol); }
    static __device__ __forceinline__ void st1(float *p, float v) { *p = v; }
    static __device__ __forceinline__ void st1_stream(float *p, float v, uint64_t pol) { st_stream_f1(p, v, pol); }
};

// a % b and ceil(a / b) for non-negative a and positive b, in 32-bit
// arithmetic when both fit (64-bit division is a long software routine)
__device__ __forceinline__ int64_t small_mod(int64_t a, int64_t b)
{
    return (a | b) <= 0xffffffffll ? static_cast<int64_t>(static_cast<uint32_t>(a) % static_cast<uint32_t>(b)) : a % b;
}

__device__ __forceinline__ int64_t small_ceil_div(int64_t a, int64_t b)
{
    const int64_t n = a + b - 1;
    return (n | b) <= 0xffffffffll ? static_cast<int64_t>(static_cast<uint32_t>(n) / static_cast<uint32_t>(b)) : n / b;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// x + o for the two bf16 values x of a packed 32-bit word (low half first):
// mixed-precision adds (sm_100 and later), which widen the bf16 operand
// exactly and round the sum once, so the result is that of widening and
// then adding in fp32, in one instruction a value.  volatile: each use
// widens again from the packed word, so a pass over a slice does not keep the
// widened values live for a later pass.
__device__ __forceinline__ float2 bf16x2_add(uint32_t w, float2 o)
{
    float a, b;
    asm volatile("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2;\n\t"
                 "add.rn.f32.bf16 %0, lo, %3;\n\tadd.rn.f32.bf16 %1, hi, %4; }"
                 : "=f"(a), "=f"(b)
                 : "r"(w), "f"(o.x), "f"(o.y));
    return make_float2(a, b);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

template <>
struct Io<__nv_bfloat16> {
    static __device__ __forceinline__ float4 unpack(uint32_t a, uint32_t b)
    {
        return make_float4(bf16_bits_to_f32(a & 0xffffu), bf16_bits_to_f32(a >> 16), bf16_bits_to_f32(b & 0xffffu),
                           bf16_bits_to_f32(b >> 16));
    }
    static __device__ __forceinline__ float4 ld4_stream(const __nv_bfloat16 *p, uint64_t pol)
    {
        uint32_t a, b;
        asm("ld.global.L1::no_allocate.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
            : "=r"(a), "=r"(b)
            : "l"(p), "l"(pol));
        return unpack(a, b);
    }
    static __device__ __forceinline__ float4 ld4_ro(const __nv_bfloat16 *p, uint64_t pol)
    {
        uint32_t a, b;
        asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
            : "=r"(a), "=r"(b)
            : "l"(p), "l"(pol));
        return unpack(a, b);
    }
    static __device__ __forceinline__ float4 ld4_param(const __nv_bfloat16 *p)
    {
        uint32_t a, b;
        asm("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "l"(p));
        return unpack(a, b);
    }
    static __device__ __forceinline__ void st4_stream(__nv_bfloat16 *p, float4 v, uint64_t pol)
    {
        asm volatile("st.global.L1::no_allocate.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(p),
                     "r"(pack_bf16x2(v.x, v.y)), "r"(pack_bf16x2(v.z, v.w)), "l"(pol)
                     : "memory");
    }
    static __device__ __forceinline__ float2 ld2_stream(const __nv_bfloat16 *p, uint64_t pol)
    {
        uint32_t a;
        asm("ld.global.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(a) : "l"(p), "l"(pol));
        return make_float2(bf16_bits_to_f32(a & 0xffffu), bf16_bits_to_f32(a >> 16));
    }
    static __device__ __forceinline__ void st2_stream(__nv_bfloat16 *p, float2 v, uint64_t pol)
    {
        asm volatile("st.global.L1::no_allocate.L2::cache_hint.u32 [%0], %1, %2;" ::"l"(p), "r"(pack_bf16x2(v.x, v.y)),
                     "l"(pol)
                     : "memory");
    }
    static __device__ __forceinline__ float ld1(const __nv_bfloat16 *p)
    {
        unsigned short h;
        asm("ld.global.u16 %0, [%1];" : "=h"(h) : "l"(p));
        return bf16_bits_to_f32(h);
    }
    static __device__ __forceinline__ float ld1_stream(const __nv_bfloat16 *p, uint64_t pol)
    {
        unsigned short h;
        asm("ld.global.L1::no_allocate.L2::cache_hint.u16 %0, [%1], %2;" : "=h"(h) : "l"(p), "l"(pol));
        return bf16_bits_to_f32(h);
    }
    static __device__ __forceinline__ void st1(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
    static __device__ __forceinline__ void st1_stream(__nv_bfloat16 *p, float v, uint64_t pol)
    {
        const __nv_bfloat16 b = __float2bfloat16_rn(v);
        const unsigned short h = *reinterpret_cast<const unsigned short *>(&b);
        asm volatile("st.global.L1::no_allocate.L2::cache_hint.u16 [%0], %1, %2;" ::"l"(p), "h"(h), "l"(pol)
                     : "memory");
    }
};

// ---------------------------------------------------------------- tensor memory
// Tensor memory (TMEM) is a 128-lane x 512-column array of 32-bit cells per
// SM.  An address is (lane << 16) | column.  A warp reaches only the 32
// lanes of its quarter: lanes 32*(w % 4) .. 32*(w % 4) + 31 for warp w of
// the CTA.  With the .32x32b shape, thread t of the warp moves the cells of
// lane (address lane) + t, N consecutive columns.  The .sync.aligned forms
// are executed by all 32 threads of the warp with the same address.

// Allocate `ncols` columns (a power of two, 32..512) for this CTA; one full
// warp executes it.  The TMEM address is written to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Free the columns again; executed by the warp that allocated them.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Order tensor-memory operations around a thread barrier.
__device__ __forceinline__ void tmem_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Store 4 columns of this thread's lane.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, float4 v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
                 "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
                 "r"(__float_as_uint(v.w))
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Load 4 columns of this thread's lane.  The registers are valid only after
// tmem_wait_ld_pin() on them.
__device__ __forceinline__ float4 tmem_ld4(uint32_t taddr)
{
    uint32_t a, b, c, d;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(taddr)
                 : "memory");
    return make_float4(__uint_as_float(a), __uint_as_float(b), __uint_as_float(c), __uint_as_float(d));
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// After tmem_wait_ld(): make every later use of v depend on the wait, so the
// compiler cannot move a use of the loaded registers above it.
__device__ __forceinline__ void tmem_pin(float4 &v)
{
    asm volatile("" : "+f"(v.x), "+f"(v.y), "+f"(v.z), "+f"(v.w));
}

// ---------------------------------------------------------------- statistics

// A partial of (count, mean, M2 = sum of squared deviations from mean).
struct Moments {
    float n, mean, m2;
};

// Chan et al. pairwise update: fold b into a.
__device__ __forceinline__ void chan_merge(Moments &a, const Moments &b)
{
    const float n = a.n + b.n;
    if (b.n == 0.f)
        return;
    const float delta = b.mean - a.mean;
    const float f = b.n / n;
    a.mean = fmaf(delta, f, a.mean);
    a.m2 = a.m2 + b.m2 + delta * delta * a.n * f;
    a.n = n;
}

__device__ __forceinline__ Moments shfl_xor_moments(const Moments &a, int lane_mask)
{
    Moments b;
    b.n = __shfl_xor_sync(0xffffffffu, a.n, lane_mask);
    b.mean = __shfl_xor_sync(0xffffffffu, a.mean, lane_mask);
    b.m2 = __shfl_xor_sync(0xffffffffu, a.m2, lane_mask);
    return b;
}

// Butterfly merge over the 32 lanes of a warp; every lane ends with the
// result.  Each step is Chan's update with the lower lane's partial (lo)
// first and the upper lane's (up) second, on both partners: n and
// lo.m2 + up.m2 are symmetric, and delta = up.mean - lo.mean is the
// partners' difference negated exactly on the upper lane, so both compute
// the same bits and the result is deterministic.
__device__ __forceinline__ Moments warp_merge(Moments a)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const Moments b = shfl_xor_moments(a, o);
        const bool upper = (lane & o) != 0;
        const float n = a.n + b.n;
        const float d = b.mean - a.mean;
        const float delta = upper ? -d : d;
        const float up_n = upper ? a.n : b.n;
        const float lo_n = upper ? b.n : a.n;
        const float lo_mean = upper ? b.mean : a.mean;
        const float f = n > 0.f ? up_n / n : 0.f;
        a.mean = fmaf(delta, f, lo_mean);
        a.m2 = (a.m2 + b.m2) + delta * delta * lo_n * f;
        a.n = n;
    }
    return a;
}

// The row mean as an unevaluated fp32 pair (hi + lo) and 1/sqrt(var + eps).
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

// Sum of v over a CTA of NT threads, in a fixed order; every thread gets the
// result.  `scratch` (NT / 32 floats) must not be in use by the previous call.
template <int NT>
__device__ __forceinline__ float block_sum(float v, float *scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0)
        scratch[warp] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w)
        t += scratch[w];
    return t;
}

// ---------------------------------------------------------------- launchers

// Launch `k` with programmatic stream serialization (see pdl_begin).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, static_cast<Args &&>(args)...);
}

// Workspace header of the LayerNorm kernels (256 bytes).  The caller zeroes
// the whole workspace before first use and after a timeout; between those,
// the persistent kernel keeps it consistent from call to call.
struct LnSync {
    unsigned row_base; // rows the persistent kernel has processed on this workspace (mod 2^32)
    unsigned done;     // CTAs of the current launch that are done with row_base
    unsigned pad[62];
};
static_assert(sizeof(LnSync) == 256, "LnSync must be 256 bytes");

// Tensors are fp32 (float) or bf16 (__nv_bfloat16) in memory; the kernel
// templated on the element type casts these.
struct LnParams {
    const void *x;
    const void *gamma; // may be null
    const void *beta;  // may be null
    void *y;
    int64_t rows;
    int64_t row_len; // elements
    float eps;
    LnSync *sync;
    float4 *part; // persistent: tagged records [slots][grid][2] (u64); split: partials [rows][P]
    unsigned *err;
    uint64_t timeout_ns;
    unsigned tag_skew; // test hook: 0, or an offset that makes the grid barrier unreachable
    int max_n4;        // float4 capacity of each shared-memory row buffer
    int groups;        // persistent: row groups (the grid is groups x CTAs per group)
    int64_t chunk;     // split: elements per CTA (multiple of 4 on the vector path)
    int parts;         // split: CTAs per row (P)
};

// Persistent single-read LayerNorm (one CTA per SM, cooperative launch).
struct LnPersistentConfig {
    int threads;              // CTA size
    int data_threads;         // threads that own the row slice
    int v4_per_thread;        // float4 of the slice per data thread
    int record_bytes_per_cta; // workspace bytes of barrier records per CTA
    int max_grid;             // most CTAs the kernel supports
};
LnPersistentConfig ln_persistent_config();
// Max dynamic shared memory the kernel may use; called once per device.
cudaError_t ln_persistent_static_smem(int *bytes);
cudaError_t ln_persistent_setup(int max_dynamic_smem);
// Number of co-resident CTAs per SM for `dyn_smem` bytes.
cudaError_t ln_persistent_occupancy(int dyn_smem, int *ctas_per_sm);
// The persistent kernel's GroupNorm form: row r is segment (r / G, r % G) of
// M channels x S positions (S a multiple of the 16-byte unit's 4 fp32 or 8
// bf16 values); gamma/beta of LnParams are per channel [G * M]; the output is
// 2 LReLU((x - mean) * rstd * gamma + beta).
struct GnPersist {
    int64_t G;
    uint32_t M, S;
    float slope;
};
// bf16: x, y, gamma, beta of bfloat16 (row_len a multiple of 8, max_n4 and
// the slices counted in 16-byte units), else fp32.  gn: null for LayerNorm,
// else the GroupNorm form over NCHW segments.
cudaError_t ln_persistent_launch(const LnParams &p, int grid, int dyn_smem, cudaStream_t stream, bool bf16,
                                 const GnPersist *gn = nullptr);

// Two-kernel LayerNorm (partials, then merge + apply); any shape.  bf16:
// the tensors are bf16, else fp32.  vec4: rows are a multiple of 4 elements
// and the pointers 4-element aligned.
cudaError_t ln_split_launch(const LnParams &p, bool bf16, bool vec4, cudaStream_t stream);
// Its first kernel alone: part[r * P + pc] = (n, mean of x - K, M2, K) of
// chunk pc of row r (K = x[r][0]).
cudaError_t ln_split_stats_launch(const LnParams &p, bool bf16, bool vec4, cudaStream_t stream);

// One-launch LayerNorm for rows of at most ln_rows_max_row_len() elements
// (a multiple of 4, 4-element aligned pointers); no workspace.
int64_t ln_rows_max_row_len();
cudaError_t ln_rows_launch(const LnParams &p, bool bf16, int sm_count, cudaStream_t stream);

// GroupNorm + LeakyReLU + x2 (bf16: the tensors are bf16, else fp32).
cudaError_t gn_vec4_launch(const void *x, const void *gamma, const void *beta, void *y, int64_t N, int64_t C,
                           int64_t M, float eps, float slope, bool bf16, int sm_count, cudaStream_t stream);

// GroupNorm + LeakyReLU + x2 over segments: x[R][L] with R = N * G segments of
// L = M * S elements; element e of segment r belongs to channel
// (r % G) * M + e / S.  The 2-D (N, C) form is S = 1.
struct GnSegParams {
    const void *x;
    const void *gamma; // [C] or null
    const void *beta;  // [C] or null
    void *y;
    int64_t rows;    // R = N * G
    int64_t seg_len; // L = M * S
    int64_t G, M, S;
    float eps, slope;
    const float4 *part; // split path: partials [R][parts] from ln_split_stats_launch
    int64_t chunk;      // split path: elements per CTA
    int parts;          // split path: CTAs per segment; register paths: cluster size
    int per4;           // streamed path: vectors per CTA slice
    int cache_gb;       // streamed path, one channel per element: read gamma/beta through L1
    uint64_t timeout_ns; // streamed path: longest mbarrier wait
    unsigned *err;       // streamed path: the device error word
};
// Segment in registers: NT threads a CTA, a cluster of `cluster` CTAs per
// segment (1, 2, 4, 8 or 16), V 4-element vectors a thread.  Needs L % 4 == 0,
// 4-element aligned pointers and L / 4 <= gns_reg_capacity4(cluster).
int64_t gns_reg_capacity4(int cluster);
// Clusters that can be co-resident (0 if the cluster size cannot launch).
cudaError_t gns_reg_max_clusters(int64_t seg_len, int64_t S, bool bf16, int cluster, int *clusters);
cudaError_t gns_reg_launch(const GnSegParams &p, bool bf16, int cluster, cudaStream_t stream);
// Streamed register path: persistent clusters, each CTA's next slice arrives
// by bulk copy into shared memory.  Needs L % 4 == 0 (L % 8 for bf16),
// 16-byte aligned x, 4-element aligned y/gamma/beta, and a slice of at most
// gns_stream_capacity4() vectors.
// act: GroupNorm's LeakyReLU x2 epilogue; without it the kernel is
// LayerNorm over rows of seg_len with per-element gamma/beta (G = 1, M = L,
// S = 1).  wide: the group is split over twice the CTAs of the smallest
// cluster that holds it (bf16 slices of 2,048 vectors then take a form sized
// for 5 CTAs per SM).
cudaError_t gns_stream_max_clusters(int64_t seg_len, int64_t S, bool bf16, bool act, int cluster, bool wide,
                                    int *clusters);
// Largest CTA slice (4-element vectors) of the streamed kernel.
int64_t gns_stream_capacity4(bool bf16);
cudaError_t gns_stream_launch(const GnSegParams &p, bool bf16, bool act, int cluster, bool wide, cudaStream_t stream);
// Apply kernel of the split path (after ln_split_stats_launch on the same
// segments); vec4 as for the LayerNorm split path.
cudaError_t gns_split_apply_launch(const GnSegParams &p, bool bf16, bool vec4, cudaStream_t stream);
// Short segments: a team of lanes per segment, up to 8 items a lane, an item
// being `elems` (4, 2 or 1) consecutive elements, so x, y and seg_len
// aligned to that many; at most gns_team_max_items() items a segment.
int64_t gns_team_max_items();
cudaError_t gns_team_launch(const GnSegParams &p, bool bf16, int elems, int sm_count, cudaStream_t stream);
// One warp per segment, scalar loads; any shape (x is re-read from L1/L2).
cudaError_t gns_warp_launch(const GnSegParams &p, bool bf16, int sm_count, cudaStream_t stream);

// Linear then GroupNorm + LeakyReLU + x2: y = 2 LReLU(GN(x W^T + bias)), x
// [Mr][K] and W [N][K] bfloat16 (K-major), bias/gamma/beta [N] fp32 or null,
// y [Mr][N] fp32; groups of `group` contiguous channels.  Needs K % 8 == 0,
// 16-byte aligned x, W and y, and linear_gn_group_size_ok(group).
struct LinGnParams {
    const void *x, *w;
    const float *bias, *gamma, *beta;
    float *y;
    int64_t Mr, K, N, group;
    float eps, slope;
    uint64_t timeout_ns;
    unsigned *err;
};
bool linear_gn_group_size_ok(int64_t group);
cudaError_t linear_gn_launch(const LinGnParams &p, int sm_count, cudaStream_t stream);

// RMSNorm over dim 1 of [B][C][S] (bf16: the tensors are bf16, else fp32).
cudaError_t rms_channel_launch(const void *x, void *y, int64_t B, int64_t C, int64_t S, float eps, bool bf16,
                               cudaStream_t stream);

} // namespace normk

namespace normapi {
// Validate a LayerNorm call on esz-byte elements (4 = fp32, 2 = bf16) and
// choose its path exactly as norm_layer_fwd would (current device, current
// options), launching nothing.  *ws_bytes = the workspace bytes that path
// uses: 0 for the row kernel and the cluster kernel, the header and tagged
// records for the persistent kernel, the header and per-chunk partials for
// the two-kernel path.  Returns the status norm_layer_fwd would return for
// the same arguments before its launch.
norm_status_t layer_fwd_workspace_need(const void *x, const void *gamma, const void *beta, const void *y,
                                       int64_t rows, int64_t row_len, float eps, int esz, size_t *ws_bytes);
} // namespace normapi
