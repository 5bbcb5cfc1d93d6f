// linear_gn_kernels.cu - the GroupNorm page's module in one kernel: the Linear
// h = x W^T + bias, then GroupNorm + LeakyReLU + x + x on each row of h
// (POPCORNBENCH transcript "Kimi-K2.6 l2_p62": the module's forward is
// F.linear followed by the fused normalization, and the first design turn
// weighs computing the group statistics in the GEMM's epilogue so that h
// never goes to memory).
//
// The contraction runs on the 5th-generation tensor cores: x and W are
// bfloat16 (K-major, as nn.Linear stores W), products are accumulated in fp32
// in tensor memory, and the epilogue is fp32.
//
// One CTA per SM walks output tiles of 256 rows x 256 channels (persistent,
// tile t -> rows (t % tiles_m) * 256, channels (t / tiles_m) * 256, so the CTAs
// running at once share W's rows through L2).  A 256-row tile is two MMA row
// halves of 128 that share every slice of W: per MMA cycle a CTA pulls 64
// bytes of operands from L2 instead of the 96 of a 128 x 256 tile, which is
// what the operand fetch of the whole GPU can sustain.  Warp roles:
//   warp 0, one lane     TMA producer: 64-wide K slices of x (256 x 64) and W
//                        (256 x 64) by cp.async.bulk.tensor, 128-byte
//                        swizzled, into a ring of LG_STAGES shared-memory
//                        stages, each tracked by a "full" mbarrier;
//   warp 1, one lane     MMA issuer: per stage, four K steps of two
//                        tcgen05.mma (M 128, N 256, K 16), one per row half,
//                        into the two halves of the TMEM accumulator (256 fp32
//                        columns each); tcgen05.commit releases the stage
//                        ("empty" mbarrier) and, after the tile's last stage,
//                        hands the accumulator to the epilogue;
//   warps 2..5           epilogue: thread t of the 128 owns rows t and 128 + t
//                        of the tile (TMEM lane t of each half).  A group of CG
//                        contiguous channels is CG consecutive TMEM columns
//                        of one lane, so each thread holds whole groups in
//                        registers: it adds the bias, takes the group's mean
//                        and then the exact M2 about it, applies gamma/beta,
//                        LeakyReLU and x + x, and stores the group's CG
//                        floats.  Then it releases the accumulator for the
//                        CTA's next tile.
// Every wait is bounded (%globaltimer): a role that gives up records
// NORM_ERR_TIMEOUT, tells the others through shared memory, and the CTA drains
// its own bulk copies and MMAs before it frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "norm_internal.cuh"

namespace normk {

namespace {

constexpr int LG_BM = 256;  // rows of x per tile: two MMA row halves
constexpr int LG_MH = 128;  // rows per MMA (M)
constexpr int LG_BN = 256;  // output channels per tile (MMA N)
constexpr int LG_BK = 64;   // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int LG_UK = 16;   // K per tcgen05.mma of kind f16
constexpr int LG_STAGES = 3;
constexpr int LG_PF = 8; // stages of W prefetched into L2 ahead of their load (measured: 113.6 -> 110.6 us)
constexpr int LG_EC = 64; // accumulator columns the epilogue loads from TMEM per wait
constexpr uint32_t LG_A_BYTES = LG_BM * LG_BK * 2;
constexpr uint32_t LG_B_BYTES = LG_BN * LG_BK * 2;
constexpr uint32_t LG_STAGE_MAX = LG_A_BYTES + LG_B_BYTES; // stage stride: the widest tile's bytes
constexpr int LG_THREADS = 192;
constexpr uint32_t LG_TMEM_COLS = 2 * LG_BN; // the accumulator: two row halves
constexpr size_t LG_SMEM = LG_STAGES * LG_STAGE_MAX + 1024; // + room to align to 1024

// Instruction descriptor of tcgen05.mma kind::f16 for N output columns: D
// fp32 (bits 4-5 = 1), A and B bfloat16 (bits 7-9, 10-12 = 1), both K-major
// (bits 15, 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__device__ __forceinline__ uint32_t mma_idesc(int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(LG_MH >> 4) << 24);
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart (the
// stride byte offset), start address >> 4 in bits 0-13, leading byte offset
// (not used by this layout) 16 bytes, descriptor version 1 in bits 46-48,
// swizzle mode 2 (128-byte) in bits 61-63.  The tile base is 1024-byte
// aligned; stepping K by 16 elements inside the 128-byte row adds 32 bytes to
// the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(16u >> 4) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// Bring a 2-D tile of the tensor into L2 ahead of its load.
__device__ __forceinline__ void tma_prefetch_l2(const CUtensorMap *map, int c0, int c1)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 16 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
                 "%13, %14, %15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

// Wait for phase `parity` of `bar`, giving up after timeout_ns or as soon as
// another role has given up (*abort set).
__device__ __forceinline__ bool lg_wait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns, volatile int *abort)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort || globaltimer_ns() - t0 > timeout_ns)
            return false;
    }
    return true;
}

struct LinGnArgs {
    const float *bias, *gamma, *beta; // [N] each, or null
    float *y;                         // [Mr][N]
    int Mr, K, N;
    int tiles_m, tiles;
    // Channel tiles: N is cut into tiles_n tiles of whole groups, as equal as
    // possible (n_base or n_base + 1 groups; the first n_extra get one more),
    // each at most LG_BN channels; W's tensor map moves w_rows rows (the
    // widest tile) per stage.
    int tiles_n, n_base, n_extra, w_rows;
    float eps, slope;
    uint64_t timeout_ns;
    unsigned *err;
};

// CG: channels per group (16, 32 or 64), a divisor of the 256-channel tile.
template <int CG>
__global__ void __launch_bounds__(LG_THREADS, 1)
    linear_gn_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                     const LinGnArgs a)
{
    extern __shared__ uint8_t lg_smem_raw[];
    __shared__ __align__(8) uint64_t full[LG_STAGES], empty[LG_STAGES];
    __shared__ __align__(8) uint64_t acc_full, acc_empty, drain;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 1024-byte aligned stages (the 128-byte swizzle repeats every 1024 bytes)
    const uint32_t raw = smem_u32(lg_smem_raw);
    uint8_t *smem = lg_smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int nk = (a.K + LG_BK - 1) / LG_BK;
    const uint32_t stage_bytes = LG_A_BYTES + static_cast<uint32_t>(a.w_rows) * LG_BK * 2;
    // channels [n0, n0 + nw) of channel tile j
    auto ntile = [&](int j, int &n0, int &nw) {
        n0 = (j * a.n_base + min(j, a.n_extra)) * CG;
        nw = (a.n_base + (j < a.n_extra ? 1 : 0)) * CG;
    };
    const uint64_t drain_ns = a.timeout_ns > 100000000ull ? a.timeout_ns : 100000000ull;
    volatile int *abort = &abort_s;

    if (warp == 1)
        tmem_alloc(&tmem_base_s, LG_TMEM_COLS);
    if (threadIdx.x == 0) {
        for (int s = 0; s < LG_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&acc_full, 1);
        mbar_init(&acc_empty, 4); // one arrival per epilogue warp
        mbar_init(&drain, 1);
        abort_s = 0;
        fence_mbar_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_x)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_w)) : "memory");
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tmem_base = tmem_base_s;
    bool failed = false;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            int64_t fills = 0; // stage fills issued so far (fill f uses stage f % LG_STAGES)
            for (int t = blockIdx.x; t < a.tiles && !failed; t += gridDim.x) {
                const int m0 = (t % a.tiles_m) * LG_BM;
                int n0, nw;
                ntile(t / a.tiles_m, n0, nw);
                for (int kb = 0; kb < nk; ++kb, ++fills) {
                    const int s = static_cast<int>(fills % LG_STAGES);
                    const uint32_t use = static_cast<uint32_t>(fills / LG_STAGES);
                    // the MMAs of this stage's previous fill have read it
                    if (!lg_wait(&empty[s], (use & 1u) ^ 1u, a.timeout_ns, abort)) {
                        failed = true;
                        break;
                    }
                    uint8_t *sa = smem + s * LG_STAGE_MAX;
                    // W's slice LG_PF stages ahead into L2, so its load finds it there
                    if (kb + LG_PF < nk)
                        tma_prefetch_l2(&map_w, (kb + LG_PF) * LG_BK, n0);
                    mbar_arrive_expect_tx(&full[s], stage_bytes);
                    tma_load_2d(sa, &map_x, kb * LG_BK, m0, &full[s]);
                    tma_load_2d(sa + LG_A_BYTES, &map_w, kb * LG_BK, n0, &full[s]);
                }
            }
            if (failed) {
                *abort = 1;
                record_error(a.err, NORM_ERR_TIMEOUT);
            }
            // Never exit with a bulk copy still writing shared memory: wait for
            // the last fill of every stage (no fill follows it).  Without a
            // failure, also wait for the MMA warp's release of those fills, so
            // that no commit arrives on an mbarrier of a CTA that has exited.
            for (int64_t f = fills - LG_STAGES > 0 ? fills - LG_STAGES : 0; f < fills; ++f) {
                const uint32_t par = static_cast<uint32_t>((f / LG_STAGES) & 1);
                if (!mbar_wait_bounded(&full[f % LG_STAGES], par, drain_ns) ||
                    (!failed && !*abort && !lg_wait(&empty[f % LG_STAGES], par, drain_ns, abort)))
                    record_error(a.err, NORM_ERR_TIMEOUT);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int64_t fills = 0;
            int local = 0; // tiles of this CTA so far
            bool issued = false;
            for (int t = blockIdx.x; t < a.tiles && !failed; t += gridDim.x, ++local) {
                // the epilogue has read the accumulator's previous tile
                if (!lg_wait(&acc_empty, (static_cast<uint32_t>(local) & 1u) ^ 1u, a.timeout_ns, abort)) {
                    failed = true;
                    break;
                }
                tmem_fence_after_sync();
                int n0, nw;
                ntile(t / a.tiles_m, n0, nw);
                const uint32_t idesc = mma_idesc(nw);
                for (int kb = 0; kb < nk; ++kb, ++fills) {
                    const int s = static_cast<int>(fills % LG_STAGES);
                    if (!lg_wait(&full[s], static_cast<uint32_t>((fills / LG_STAGES) & 1), a.timeout_ns, abort)) {
                        failed = true;
                        break;
                    }
                    tmem_fence_after_sync();
                    const uint32_t sa = smem_u32(smem + s * LG_STAGE_MAX);
#pragma unroll
                    for (int k = 0; k < LG_BK / LG_UK; ++k) {
                        const uint32_t koff = static_cast<uint32_t>(k * LG_UK * 2);
                        const uint64_t bdesc = sw128_desc(sa + LG_A_BYTES + koff);
                        const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
#pragma unroll
                        for (int h = 0; h < LG_BM / LG_MH; ++h)
                            mma_bf16(tmem_base + static_cast<uint32_t>(h * LG_BN),
                                     sw128_desc(sa + static_cast<uint32_t>(h * LG_MH * LG_BK * 2) + koff), bdesc, idesc,
                                     acc);
                    }
                    issued = true;
                    mma_commit(&empty[s]); // the stage is free once these MMAs have read it
                }
                if (failed)
                    break;
                mma_commit(&acc_full); // the tile's sums are complete
            }
            if (failed) {
                *abort = 1;
                record_error(a.err, NORM_ERR_TIMEOUT);
                // every MMA issued has finished reading shared memory and
                // writing TMEM before the CTA frees them
                if (issued) {
                    mma_commit(&drain);
                    if (!mbar_wait_bounded(&drain, 0, drain_ns))
                        record_error(a.err, NORM_ERR_TIMEOUT);
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3; // TMEM lane quarter of this warp
        int local = 0;
        for (int t = blockIdx.x; t < a.tiles; t += gridDim.x, ++local) {
            if (!lg_wait(&acc_full, static_cast<uint32_t>(local) & 1u, a.timeout_ns, abort)) {
                *abort = 1;
                record_error(a.err, NORM_ERR_TIMEOUT);
                break;
            }
            tmem_fence_after_sync();
            const int m0 = (t % a.tiles_m) * LG_BM;
            int n0, nw;
            ntile(t / a.tiles_m, n0, nw);
#pragma unroll 1
            for (int h = 0; h < LG_BM / LG_MH; ++h) {
                const int row = m0 + h * LG_MH + 32 * q + lane; // TMEM lane 32 q + lane of half h
                const uint32_t tacc =
                    tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(h * LG_BN);
                float *yr = a.y + static_cast<int64_t>(row) * a.N;
                // LG_EC columns (several groups) are loaded from TMEM with one
                // wait, so the loads' latency is paid once per chunk
#pragma unroll 1
                for (int e0 = 0; e0 < nw; e0 += LG_EC) {
                    float v[LG_EC];
#pragma unroll
                    for (int j = 0; j < LG_EC; j += 16) {
                        float w[16];
                        if (e0 + j < nw) { // the same for the whole warp
                            tmem_ld16(tacc + static_cast<uint32_t>(e0 + j), w);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                w[i] = 0.f;
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            v[j + i] = w[i];
                    }
                    tmem_wait_ld();
#pragma unroll
                    for (int gg = 0; gg < LG_EC; gg += CG) {
                        const int c0 = n0 + e0 + gg;
                        if (e0 + gg >= nw || c0 >= a.N) // past the tile (or the last channel)
                            continue;
                        // h = x W^T + bias, then the group's mean and exact M2 about it
                        float s = 0.f;
#pragma unroll
                        for (int j = 0; j < CG; ++j) {
                            v[gg + j] += a.bias ? __ldg(a.bias + c0 + j) : 0.f;
                            s += v[gg + j];
                        }
                        const float mean = s * (1.0f / CG);
                        float m2 = 0.f;
#pragma unroll
                        for (int j = 0; j < CG; ++j) {
                            const float d = v[gg + j] - mean;
                            m2 = fmaf(d, d, m2);
                        }
                        const float rstd = rsqrtf(m2 * (1.0f / CG) + a.eps);
                        if (row < a.Mr) {
#pragma unroll
                            for (int j = 0; j < CG; j += 4) {
                                float o[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const float gw = a.gamma ? __ldg(a.gamma + c0 + j + i) : 1.f;
                                    const float bw = a.beta ? __ldg(a.beta + c0 + j + i) : 0.f;
                                    float u = fmaf((v[gg + j + i] - mean) * rstd, gw, bw);
                                    u = u > 0.f ? u : a.slope * u;
                                    o[i] = u + u;
                                }
                                *reinterpret_cast<float4 *>(yr + c0 + j) = make_float4(o[0], o[1], o[2], o[3]);
                            }
                        }
                    }
                }
            }
            // this warp has read the accumulator: the MMA warp may refill it
            tmem_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&acc_empty);
        }
    }
    tmem_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tmem_fence_after_sync();
        tmem_dealloc(tmem_base, LG_TMEM_COLS);
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link to
// libcuda); looked up once.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// A [rows][K] bfloat16 K-major operand as 64 x box_rows tiles with the
// 128-byte swizzle; elements past the tensor's edge read as zero.
bool encode_operand(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, uint32_t box_rows)
{
    const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2u};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(LG_BK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int CG>
cudaError_t launch_cg(const CUtensorMap &mx, const CUtensorMap &mw, const LinGnArgs &a, int grid, cudaStream_t stream)
{
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(linear_gn_kernel<CG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(LG_SMEM));
    });
    if (attr != cudaSuccess)
        return attr;
    linear_gn_kernel<CG><<<grid, LG_THREADS, LG_SMEM, stream>>>(mx, mw, a);
    return cudaGetLastError();
}

} // namespace

bool linear_gn_group_size_ok(int64_t cg)
{
    return cg == 16 || cg == 32 || cg == 64;
}

// Channel tiling: the number of channel tiles T (each of whole groups, at
// most LG_BN channels) that minimizes the waves of tiles on the SMs times the
// widest tile, i.e. the work of the busiest SM; ties go to fewer tiles.  At
// (1024, 8192) with groups of 16: 37 tiles of 224 or 208 channels per
// 256-row block, 148 CTAs, instead of 32 tiles of 256 on 128.
static void plan_channels(int64_t tiles_m, int64_t N, int64_t cg, int sm_count, LinGnArgs *a)
{
    const int64_t units = N / cg, per_max = LG_BN / cg;
    const int64_t t_min = (units + per_max - 1) / per_max;
    int64_t best_t = t_min, best_cost = -1;
    for (int64_t t = t_min; t <= units && t <= 4 * t_min + 8; ++t) {
        const int64_t waves = (tiles_m * t + sm_count - 1) / sm_count;
        const int64_t width = (units + t - 1) / t;
        const int64_t cost = waves * width;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_t = t;
        }
    }
    a->tiles_n = static_cast<int>(best_t);
    a->n_base = static_cast<int>(units / best_t);
    a->n_extra = static_cast<int>(units % best_t);
    a->w_rows = static_cast<int>((a->n_base + (a->n_extra ? 1 : 0)) * cg);
}

cudaError_t linear_gn_launch(const LinGnParams &p, int sm_count, cudaStream_t stream)
{
    LinGnArgs a;
    a.bias = p.bias;
    a.gamma = p.gamma;
    a.beta = p.beta;
    a.y = p.y;
    a.Mr = static_cast<int>(p.Mr);
    a.K = static_cast<int>(p.K);
    a.N = static_cast<int>(p.N);
    a.tiles_m = static_cast<int>((p.Mr + LG_BM - 1) / LG_BM);
    plan_channels(a.tiles_m, p.N, p.group, sm_count, &a);
    const int64_t tiles = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
    if (tiles > 0x7fffffff)
        return cudaErrorInvalidValue;
    a.tiles = static_cast<int>(tiles);
    a.eps = p.eps;
    a.slope = p.slope;
    a.timeout_ns = p.timeout_ns;
    a.err = p.err;
    CUtensorMap mx, mw;
    if (!encode_operand(&mx, p.x, p.Mr, p.K, LG_BM) ||
        !encode_operand(&mw, p.w, p.N, p.K, static_cast<uint32_t>(a.w_rows)))
        return cudaErrorInvalidValue;
    const int grid = a.tiles < sm_count ? a.tiles : sm_count;
    switch (p.group) {
    case 16: return launch_cg<16>(mx, mw, a, grid, stream);
    case 32: return launch_cg<32>(mx, mw, a, grid, stream);
    case 64: return launch_cg<64>(mx, mw, a, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace normk
