// norm_api.cu - the extern "C" entry points declared in include/norm.h:
// argument validation (always before any CUDA call), per-device state,
// LayerNorm path planning, the device error word, and options.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "norm_internal.cuh"

// Per-device error words, one per stream slot: a launch on a stream records
// its first device-side failure (NORM_ERR_TIMEOUT) in that stream's word, and
// norm_last_error(stream) reads and clears only that word.  Slot 0 is shared
// by the streams beyond the first kErrSlots - 1 a device sees.
constexpr int kErrSlots = 256;
__device__ unsigned g_norm_error_words[kErrSlots];

namespace {

using normk::LnParams;

constexpr int kMaxDevices = 64;
constexpr size_t kWsHeader = sizeof(normk::LnSync);
// Shortest row for which the automatic choice takes the persistent kernel
// (fp32): rows past the cluster kernel's.  Rows shorter than about 1.6 Mi
// elements are split over row groups (persistent_groups) so that each
// group's row streams long enough to hide its grid exchange.
constexpr int64_t kPersistentMinRowLen = 131073;
// Rows of 32,768 to 131,072 elements take the persistent kernel (in row
// groups) rather than the cluster kernel once x holds 96 MiB or more.
// Measured on GB300 over 256 MiB of fp32 x (fraction of the copy peak):
// rows of 32,768 0.81 vs 0.73, 65,536 0.85 vs 0.74, 131,072 0.86 vs 0.73;
// bf16 over 128 MiB: 0.58 vs 0.57, 0.58 vs 0.45, 0.62 vs 0.52.  Below about
// 60-100 MiB the persistent kernel's prologue (about 5 us more than the
// cluster kernel's launch) outweighs its faster streaming.  Rows of 16,384
// stay on the row and cluster kernels (fp32 0.84 vs 0.81 persistent).
constexpr int64_t kPersistentMidRowLen = 32768;
constexpr size_t kPersistentMidMinBytes = size_t(96) << 20;
// Rows of 131,073 to 1,048,575 elements over less than 24 MiB of x take the
// two-kernel path, whose second read of x then comes from L2: measured on
// GB300 (two-kernel vs persistent, us) fp32 (8, 262144) 10.8 vs 12.3,
// (16, 262144) 15.3 vs 19.0, (32, 262144) 23.4 vs 24.3 (left to the
// persistent kernel), (48, 262144) 31.7 vs 28.0; bf16 (16, 262144) 12.8 vs
// 13.6, (32, 262144) 18.2 vs 19.9, (64, 262144) 28.7 vs 26.4.  Rows of 1 Mi
// or more stay persistent at any size (fp32 (4, 1048576) 16.7 vs 16.4).
constexpr size_t kPersistentSmallBytes = size_t(24) << 20;
constexpr int64_t kPersistentAnySizeRowLen = int64_t(1) << 20;
// NORM_OPT_LN_PATH value of the streamed cluster kernel, and the longest
// row the automatic choice gives the row kernel.  Measured on GB300 (GB/s
// fractions of the copy peak): the row kernel, its CTA sized to the row,
// runs rows of 256 to 8,192 at 0.88-0.93 (fp32) and 0.55-0.69 (bf16), ahead
// of the cluster kernel (0.78 fp32, 0.55 bf16 at 8,192); rows of 16,384 to
// 131,072 run best on the cluster kernel (fp32 0.79 to 0.70, bf16 0.58 to
// 0.48, vs 0.52 and 0.43 to 0.37 on the two-kernel path), except fp32 rows
// of 16,384 (below).
constexpr int64_t kLnStream = 4;
constexpr int64_t kLnRowsMaxAuto = 8192;
// fp32 rows of 16,384 run a little faster on the row kernel's 512-thread form
// (0.81 vs 0.79 on the cluster kernel); bf16 ones on the cluster kernel.
constexpr int64_t kLnRowsMaxAutoF32 = 16384;
// Longest row the automatic choice gives the cluster kernel: bf16 rows of
// 262,144 (which it can hold) measured faster on the two-kernel path.
constexpr int64_t kLnStreamMaxAuto = 131072;
// Largest gamma (and beta) in bytes for which the cluster kernel reads them
// through L1: the CTAs on one SM belong to different clusters and may each
// hold a different part of gamma/beta.  Measured: L1 reads help up to rows of
// 32,768 fp32 / 65,536 bf16 (fp32 rows of 16,384: 0.74 -> 0.80 of peak) and
// cost a little beyond (fp32 rows of 131,072: 0.70 -> 0.67).
constexpr size_t kGbL1Bytes = size_t(128) << 10;

struct DeviceState {
    bool init = false;
    bool ok = false;
    int sm_count = 0;
    int smem_optin = 0;
    int coop = 0;
    int ln_max_dyn_smem = 0; // dynamic smem the persistent kernel may use
    int ln_ctas_per_sm = 0;  // at the full dynamic smem budget
    unsigned *err = nullptr; // kErrSlots words
    std::unordered_map<cudaStream_t, int> err_slot; // stream -> its error word
    int err_next = 1;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    void *gn_ws = nullptr; // GroupNorm split-path partials (never shared with LayerNorm)
    size_t gn_ws_bytes = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

std::atomic<int64_t> g_opt_ln_path{0};
std::atomic<int64_t> g_opt_timeout_ns{200000000};
std::atomic<int64_t> g_opt_extra_arrivals{0};
std::atomic<int64_t> g_opt_ln_ctas{0};
std::atomic<int64_t> g_opt_gn_path{0};
std::atomic<int64_t> g_opt_gn_cluster{0};

// Resolve (and on first use initialize) the state of the current device.
norm_status_t device_state(DeviceState **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return NORM_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &s = g_dev[dev];
    if (!s.init) {
        s.init = true;
        s.ok = false;
        if (cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&s.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&s.coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) {
            cudaGetLastError();
            return NORM_ERR_CUDA;
        }
        void *err = nullptr;
        if (cudaGetSymbolAddress(&err, g_norm_error_words) != cudaSuccess) {
            cudaGetLastError();
            return NORM_ERR_CUDA;
        }
        s.err = static_cast<unsigned *>(err);
        // Dynamic shared memory of the persistent kernel: what the opt-in
        // limit leaves beside its static shared memory (barriers, reduction
        // scratch, the fetched records).
        int static_smem = 0;
        s.ln_max_dyn_smem = 0;
        if (normk::ln_persistent_static_smem(&static_smem) == cudaSuccess)
            s.ln_max_dyn_smem = s.smem_optin - static_smem;
        if (s.ln_max_dyn_smem <= 0 || normk::ln_persistent_setup(s.ln_max_dyn_smem) != cudaSuccess ||
            normk::ln_persistent_occupancy(s.ln_max_dyn_smem, &s.ln_ctas_per_sm) != cudaSuccess) {
            cudaGetLastError();
            s.ln_ctas_per_sm = 0;
        }
        s.ok = true;
    }
    if (!s.ok)
        return NORM_ERR_CUDA;
    *out = &s;
    return NORM_OK;
}

// The error word of launches on `stream` (a slot assigned on first use).
unsigned *stream_err(DeviceState &d, cudaStream_t stream)
{
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = d.err_slot.find(stream);
    if (it != d.err_slot.end())
        return d.err + it->second;
    int slot = 0;
    if (d.err_next < kErrSlots)
        slot = d.err_next++;
    d.err_slot.emplace(stream, slot);
    return d.err + slot;
}

// The library-owned workspace of `bytes` or more at *ws (of *ws_bytes bytes),
// grown stream-ordered on `stream`: the old buffer is freed and a new one
// allocated and zero-filled with cudaFreeAsync / cudaMallocAsync /
// cudaMemsetAsync, so no call synchronizes the device.  Callers serialize the
// calls that use it.  Growth is refused (NORM_ERR_WORKSPACE) while `stream`
// is being captured into a CUDA graph: an allocation made inside a capture
// belongs to the graph.
norm_status_t grow_library_workspace(void **ws, size_t *ws_bytes, size_t bytes, bool zero, cudaStream_t stream)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (*ws_bytes >= bytes)
        return NORM_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
    }
    if (cs != cudaStreamCaptureStatusNone)
        return NORM_ERR_WORKSPACE;
    if (*ws && cudaFreeAsync(*ws, stream) != cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
    }
    *ws = nullptr;
    *ws_bytes = 0;
    void *p = nullptr;
    if (cudaMallocAsync(&p, bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
    }
    if (zero && cudaMemsetAsync(p, 0, bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        cudaFreeAsync(p, stream);
        return NORM_ERR_CUDA;
    }
    *ws = p;
    *ws_bytes = bytes;
    return NORM_OK;
}

bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// [a, a+na) and [b, b+nb) in bytes intersect.
bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0)
        return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

bool valid_eps(float eps)
{
    return std::isfinite(eps) && eps >= 0.f;
}

// Product of non-negative extents without overflow of the byte count.
bool safe_mul(int64_t a, int64_t b, int64_t *out)
{
    if (a < 0 || b < 0)
        return false;
    if (a != 0 && b > (int64_t(1) << 60) / a)
        return false;
    *out = a * b;
    return true;
}

// ------------------------------------------------------------------ LN plan

struct LnPlan {
    int path = 0; // 1 persistent, 2 split
    int grid = 0;
    int groups = 1; // persistent: row groups
    int max_n4 = 0;
    int dyn_smem = 0;
    int parts = 0;
    int64_t chunk = 0;
    bool vec4 = false;
    size_t ws_bytes = 0;
};

void plan_split(int64_t rows, int64_t L, bool vec4, const DeviceState &d, LnPlan *pl)
{
    const int64_t target = int64_t(4) * d.sm_count;
    int64_t P = (target + rows - 1) / rows;
    const int64_t maxP = (L + 4095) / 4096;
    if (P > maxP)
        P = maxP;
    if (P < 1)
        P = 1;
    int64_t chunk = (L + P - 1) / P;
    if (vec4)
        chunk = (chunk + 3) & ~int64_t(3);
    P = (L + chunk - 1) / chunk;
    pl->path = 2;
    pl->vec4 = vec4;
    pl->parts = static_cast<int>(P);
    pl->chunk = chunk;
    pl->ws_bytes = kWsHeader + static_cast<size_t>(rows) * static_cast<size_t>(P) * 16u;
}

// CTAs of the persistent kernel on this device.
int persistent_grid(const DeviceState &d)
{
    const normk::LnPersistentConfig cfg = normk::ln_persistent_config();
    int grid = d.sm_count * d.ln_ctas_per_sm;
    const int64_t want = g_opt_ln_ctas.load();
    if (want > 0 && want < grid)
        grid = static_cast<int>(want);
    if (grid > cfg.max_grid)
        grid = cfg.max_grid;
    return grid;
}

// Largest per-CTA slice (float4) the persistent kernel holds: the data
// threads' share, and two row buffers in dynamic shared memory.
int64_t persistent_max_slice(const DeviceState &d)
{
    const normk::LnPersistentConfig cfg = normk::ln_persistent_config();
    int64_t m = int64_t(cfg.data_threads) * cfg.v4_per_thread;
    const int64_t by_smem = (d.ln_max_dyn_smem / 32) / 8 * 8; // two buffers, 128-byte rounded
    return m < by_smem ? m : by_smem;
}

// Longest row of esz-byte elements the persistent kernel serves with one HBM
// read of x: every CTA's slice of 16-byte units fits its shared-memory
// buffers, and the kernel partitions rows with 32-bit arithmetic (units per
// row * (grid + 1) < 2^32, elements of a row < 2^32).
int64_t persistent_max_row_len(const DeviceState &d, int esz = 4)
{
    if (!d.coop || d.ln_ctas_per_sm < 1)
        return 0;
    const int64_t ue = 16 / esz; // elements per unit
    const int grid = persistent_grid(d);
    const int64_t by_slice = persistent_max_slice(d) * grid * ue;
    const int64_t by_index = ((int64_t(1) << 32) - 1) / (grid + 1) * ue;
    int64_t m = by_slice < by_index ? by_slice : by_index;
    if (m > (int64_t(1) << 31))
        m = int64_t(1) << 31;
    return m / ue * ue;
}

// Row groups of the persistent kernel for `rows` rows of L elements of esz
// bytes on a grid of at most gmax CTAs, or 0 if no split of the grid holds a
// row slice.  A group's CTAs must hold its slices (at most max_slice 16-byte
// units each), and a group's row must stream for about 5.5 us or more at
// the HBM rate (5.5 us * 6.5 TB/s / (2 esz bytes an element) = 18,000,000 /
// (esz L) groups at least; 4,500,000 / L for fp32) so that the grid
// exchange, two rows ahead, hides behind it.  Measured on GB300 (fraction
// of the copy peak): 2.6 us a group row gave 0.73-0.76, 3.9-5.2 us 0.87-0.92;
// (256, 262144) took 92.7 us in 15 groups against 93.5 us in the 13 that a
// 4 us floor gives, other shapes within 0.3 us.  Among the admissible
// counts (at most one group per row), the one that leaves the fewest idle
// row slots (ceil(rows / k) * k) wins; ties go to more groups.
int persistent_groups(int64_t rows, int64_t L, int gmax, int64_t max_slice, int esz)
{
    const int64_t Lu = L * esz / 16;
    const int64_t gk_min = (Lu + max_slice - 1) / max_slice;
    if (gk_min < 1 || gk_min > gmax)
        return 0;
    int64_t kmax = gmax / gk_min;
    if (kmax > rows)
        kmax = rows;
    const int64_t per_group_bytes = int64_t(18000000) / esz; // elements x esz
    int64_t kmin = (per_group_bytes + L - 1) / L;
    if (kmin < 1)
        kmin = 1;
    if (kmin > kmax)
        kmin = kmax;
    int64_t best = kmin, best_slots = (rows + kmin - 1) / kmin * kmin;
    for (int64_t k = kmin + 1; k <= kmax; ++k) {
        const int64_t slots = (rows + k - 1) / k * k;
        if (slots <= best_slots) {
            best = k;
            best_slots = slots;
        }
    }
    return static_cast<int>(best);
}

// Fills the persistent plan for rows of L elements of esz bytes (4 fp32, 2
// bf16) if the shape qualifies (whole 16-byte units); returns false if not.
bool plan_persistent(int64_t rows, int64_t L, const DeviceState &d, LnPlan *pl, int esz = 4)
{
    const int64_t ue = 16 / esz;
    if (L % ue != 0 || L > persistent_max_row_len(d, esz) || rows < 1)
        return false;
    const normk::LnPersistentConfig cfg = normk::ln_persistent_config();
    const int gmax = persistent_grid(d);
    const int groups = persistent_groups(rows, L, gmax, persistent_max_slice(d), esz);
    if (groups < 1)
        return false;
    const int gk = gmax / groups;
    const int grid = gk * groups;
    const int64_t Lu = L / ue;
    int64_t max_n4 = (Lu + gk - 1) / gk;
    if (max_n4 < 1)
        max_n4 = 1;
    pl->path = 1;
    pl->vec4 = true;
    pl->grid = grid;
    pl->groups = groups;
    pl->max_n4 = static_cast<int>(max_n4);
    pl->dyn_smem = static_cast<int>(2 * ((max_n4 + 7) / 8 * 8) * 16);
    pl->ws_bytes = kWsHeader + static_cast<size_t>(cfg.record_bytes_per_cta) * static_cast<size_t>(grid);
    return true;
}

// ------------------------------------------------------------------ GN plan

// Segment GroupNorm paths (NORM_OPT_GN_PATH values).
constexpr int kGnReg = 1, kGnSplit = 2, kGnWarp = 3, kGnStream = 4, kGnTeam = 5, kGnPersistent = 6;
// Shortest CTA slice (vectors) for which the automatic choice streams.
constexpr int64_t kGnStreamMinPer = 256;
// Longest non-vector segment the warp path takes on its own.
constexpr int64_t kGnWarpMaxLen = 4096;
// Smallest x (bytes) for which the automatic choice takes the persistent path
// over the two-kernel one: below it the second read of x mostly hits L2.
// Measured on GB300 with segments of 262,144 and 1,048,576 values: 33.5 MB
// of x took 20.8-21.5 us by two kernels and 22.2-24.9 us persistent; 67 MB
// took 39.3 and 35.6 us; 134 MB 66.2 and 56.6 us.
constexpr size_t kGnPersistentMinBytes = size_t(48) << 20;

struct GnPlan {
    int path = 0;
    bool vec4 = false;
    int parts = 0;
    int64_t chunk = 0;
    size_t ws_bytes = 0;
};

// Smallest cluster whose CTAs each hold at most a full CTA slice.
int gn_auto_cluster(int64_t L4)
{
    for (int cl = 1; cl <= 16; cl <<= 1)
        if ((L4 + cl - 1) / cl <= normk::gns_reg_capacity4(1))
            return cl;
    return 0;
}

// Smallest cluster whose streamed-kernel slices (an even number of vectors)
// hold at most cap vectors each; 0 if none of 1..16 does.
int stream_auto_cluster(int64_t L4, int64_t cap)
{
    for (int cl = 1; cl <= 16; cl <<= 1) {
        int64_t per = (L4 + cl - 1) / cl;
        per = (per + 1) & ~int64_t(1);
        if (per <= cap)
            return cl;
    }
    return 0;
}

// Offset of the split path's partials in a GroupNorm workspace: past the
// header and records of the persistent path at its largest grid, so that
// neither path overwrites what the other keeps there.
size_t gn_split_offset()
{
    const normk::LnPersistentConfig cfg = normk::ln_persistent_config();
    const size_t b = kWsHeader + static_cast<size_t>(cfg.record_bytes_per_cta) * static_cast<size_t>(cfg.max_grid);
    return (b + 255) & ~size_t(255);
}

// Partials of the split path: R * P triples after gn_split_offset(); P as the
// LayerNorm split path.
void plan_gn_split(int64_t R, int64_t L, bool vec4, const DeviceState &d, GnPlan *pl)
{
    LnPlan lp;
    plan_split(R, L, vec4, d, &lp);
    pl->path = kGnSplit;
    pl->vec4 = vec4;
    pl->parts = lp.parts;
    pl->chunk = lp.chunk;
    pl->ws_bytes = gn_split_offset() + static_cast<size_t>(R) * static_cast<size_t>(lp.parts) * 16u;
}

// Upper bound of plan_gn_split's workspace over both vector forms.
size_t gn_split_ws_bound(int64_t R, int64_t L, const DeviceState &d)
{
    GnPlan a, b;
    plan_gn_split(R, L, false, d, &a);
    plan_gn_split(R, L, true, d, &b);
    return a.ws_bytes > b.ws_bytes ? a.ws_bytes : b.ws_bytes;
}

} // namespace

extern "C" {

const char *norm_status_string(norm_status_t s)
{
    switch (s) {
    case NORM_OK: return "NORM_OK";
    case NORM_ERR_INVALID_ARG: return "NORM_ERR_INVALID_ARG";
    case NORM_ERR_MISALIGNED: return "NORM_ERR_MISALIGNED";
    case NORM_ERR_WORKSPACE: return "NORM_ERR_WORKSPACE";
    case NORM_ERR_CUDA: return "NORM_ERR_CUDA";
    case NORM_ERR_TIMEOUT: return "NORM_ERR_TIMEOUT";
    case NORM_ERR_UNSUPPORTED: return "NORM_ERR_UNSUPPORTED";
    }
    return "NORM_ERR_UNKNOWN";
}

norm_status_t norm_set_option(norm_option_t option, int64_t value)
{
    if (value < 0)
        return NORM_ERR_INVALID_ARG;
    switch (option) {
    case NORM_OPT_LN_PATH:
        if (value > 4)
            return NORM_ERR_INVALID_ARG;
        g_opt_ln_path = value;
        return NORM_OK;
    case NORM_OPT_BARRIER_TIMEOUT_NS:
        if (value == 0)
            return NORM_ERR_INVALID_ARG;
        g_opt_timeout_ns = value;
        return NORM_OK;
    case NORM_OPT_BARRIER_EXTRA_ARRIVALS:
        if (value > 1024)
            return NORM_ERR_INVALID_ARG;
        g_opt_extra_arrivals = value;
        return NORM_OK;
    case NORM_OPT_LN_CTAS:
        g_opt_ln_ctas = value;
        return NORM_OK;
    case NORM_OPT_GN_PATH:
        if (value > 6)
            return NORM_ERR_INVALID_ARG;
        g_opt_gn_path = value;
        return NORM_OK;
    case NORM_OPT_GN_CLUSTER:
        if (value > 16 || (value & (value - 1)) != 0)
            return NORM_ERR_INVALID_ARG;
        g_opt_gn_cluster = value;
        return NORM_OK;
    }
    return NORM_ERR_INVALID_ARG;
}

int64_t norm_get_option(norm_option_t option)
{
    switch (option) {
    case NORM_OPT_LN_PATH: return g_opt_ln_path.load();
    case NORM_OPT_BARRIER_TIMEOUT_NS: return g_opt_timeout_ns.load();
    case NORM_OPT_BARRIER_EXTRA_ARRIVALS: return g_opt_extra_arrivals.load();
    case NORM_OPT_LN_CTAS: return g_opt_ln_ctas.load();
    case NORM_OPT_GN_PATH: return g_opt_gn_path.load();
    case NORM_OPT_GN_CLUSTER: return g_opt_gn_cluster.load();
    }
    return -1;
}

size_t norm_layer_workspace_bytes(int64_t rows, int64_t row_len)
{
    if (rows <= 0 || row_len <= 0)
        return kWsHeader;
    DeviceState *d = nullptr;
    if (device_state(&d) != NORM_OK)
        return 0;
    LnPlan ps, pp;
    plan_split(rows, row_len, (row_len & 3) == 0, *d, &ps);
    size_t bytes = ps.ws_bytes;
    // the persistent plan of either element type (the call does not say which)
    for (int esz = 4; esz >= 2; esz -= 2) {
        if (plan_persistent(rows, row_len, *d, &pp, esz) && pp.ws_bytes > bytes)
            bytes = pp.ws_bytes;
    }
    return bytes;
}

int64_t norm_layer_max_resident_row_len(void)
{
    DeviceState *d = nullptr;
    if (device_state(&d) != NORM_OK)
        return 0;
    return persistent_max_row_len(*d);
}

norm_status_t norm_layer_workspace_reset(void *workspace, size_t bytes, cudaStream_t stream)
{
    if (!workspace || bytes < kWsHeader)
        return NORM_ERR_INVALID_ARG;
    if (cudaMemsetAsync(workspace, 0, bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
    }
    return NORM_OK;
}

} // extern "C"

namespace {

// The path a LayerNorm call takes and what it needs.
struct LnChoice {
    bool persistent = false, row_kernel = false, ln_stream = false;
    int ln_cluster = 0; // CTAs per row of the cluster kernel
    LnPlan pl;          // ws_bytes: the workspace the path uses (0 for none)
};

// Validate a LayerNorm call on tensors of esz-byte elements (4 = fp32, 2 =
// bf16) and choose its path for the current device and options, launching
// nothing.  *empty is set when the call has no elements (a no-op).
norm_status_t layer_plan(const void *x, const void *gamma, const void *beta, const void *y, int64_t rows,
                         int64_t row_len, float eps, const void *workspace, size_t workspace_bytes, int esz,
                         DeviceState **dev, LnChoice *ch, bool *empty)
{
    const bool bf16 = esz == 2;
    int64_t n = 0;
    *empty = false;
    if (rows < 0 || row_len < 0 || !valid_eps(eps) || !safe_mul(rows, row_len, &n))
        return NORM_ERR_INVALID_ARG;
    if (n == 0) {
        *empty = true;
        return NORM_OK;
    }
    if (!x || !y)
        return NORM_ERR_INVALID_ARG;
    if (!aligned(x, esz) || !aligned(y, esz) || !aligned(gamma, esz) || !aligned(beta, esz))
        return NORM_ERR_MISALIGNED;
    const size_t nb = static_cast<size_t>(n) * esz, pb = static_cast<size_t>(row_len) * esz;
    if ((x != y && overlaps(x, nb, y, nb)) || overlaps(gamma, pb, y, nb) || overlaps(beta, pb, y, nb))
        return NORM_ERR_INVALID_ARG;
    if (workspace && (!aligned(workspace, 256) || overlaps(workspace, workspace_bytes, y, nb) ||
                      overlaps(workspace, workspace_bytes, x, nb)))
        return NORM_ERR_WORKSPACE;

    DeviceState *d = nullptr;
    norm_status_t st = device_state(&d);
    if (st != NORM_OK)
        return st;
    *dev = d;

    const uintptr_t va = 4u * esz; // alignment of a 4-element vector
    const bool vec4 = (row_len & 3) == 0 && aligned(x, va) && aligned(y, va) && aligned(gamma, va) &&
                      aligned(beta, va);
    const int64_t path_opt = g_opt_ln_path.load();
    LnChoice c;
    // Streamed cluster kernel (shared with GroupNorm: one group per row, no
    // activation): rows of up to 131,072 elements, read once.
    if (vec4 && aligned(x, 16) && (bf16 ? (row_len & 7) == 0 : true)) {
        const int cl = stream_auto_cluster(row_len / 4, normk::gns_stream_capacity4(bf16));
        int active = 0;
        if (cl && normk::gns_stream_max_clusters(row_len, 1, bf16, false, cl, false, &active) == cudaSuccess && active >= 1)
            c.ln_cluster = cl;
        else
            cudaGetLastError();
    }
    if (path_opt == kLnStream && !c.ln_cluster)
        return NORM_ERR_UNSUPPORTED;
    // the persistent kernel moves whole 16-byte units (4 fp32 or 8 bf16
    // values) of 16-byte aligned tensors
    const bool unit_ok = row_len % (16 / esz) == 0 && aligned(x, 16) && aligned(y, 16) && aligned(gamma, 16) &&
                         aligned(beta, 16);
    const bool pers_wanted =
        path_opt == 1 ||
        (path_opt == 0 &&
         ((row_len >= kPersistentMinRowLen && (nb >= kPersistentSmallBytes || row_len >= kPersistentAnySizeRowLen)) ||
          (row_len >= kPersistentMidRowLen && nb >= kPersistentMidMinBytes)));
    LnPlan pp;
    if (pers_wanted && unit_ok && plan_persistent(rows, row_len, *d, &pp, esz)) {
        c.pl = pp;
        c.persistent = true;
    }
    if (path_opt == 1 && !c.persistent)
        return NORM_ERR_UNSUPPORTED;
    const int64_t rows_max_auto = bf16 ? kLnRowsMaxAuto : kLnRowsMaxAutoF32;
    c.ln_stream = !c.persistent && c.ln_cluster &&
                  (path_opt == kLnStream ||
                   (path_opt == 0 && row_len > rows_max_auto && row_len <= kLnStreamMaxAuto));
    const bool row_kernel_fits = vec4 && row_len <= normk::ln_rows_max_row_len();
    c.row_kernel = !c.persistent && !c.ln_stream && row_kernel_fits &&
                   (path_opt == 3 || (path_opt == 0 && row_len < kPersistentMinRowLen));
    if (path_opt == 3 && !c.row_kernel)
        return NORM_ERR_UNSUPPORTED;
    if (c.row_kernel || c.ln_stream) {
        c.pl.path = c.ln_stream ? kLnStream : 3;
        c.pl.ws_bytes = 0;
    }
    if (!c.persistent && !c.row_kernel && !c.ln_stream)
        plan_split(rows, row_len, vec4, *d, &c.pl);
    *ch = c;
    return NORM_OK;
}

// LayerNorm on tensors of esz-byte elements: 4 = fp32, 2 = bf16.
norm_status_t layer_fwd(const void *x, const void *gamma, const void *beta, void *y, int64_t rows, int64_t row_len,
                        float eps, void *workspace, size_t workspace_bytes, cudaStream_t stream, int esz)
{
    const bool bf16 = esz == 2;
    DeviceState *d = nullptr;
    LnChoice ch;
    bool empty = false;
    norm_status_t st = layer_plan(x, gamma, beta, y, rows, row_len, eps, workspace, workspace_bytes, esz, &d, &ch,
                                  &empty);
    if (st != NORM_OK || empty)
        return st;
    const LnPlan &pl = ch.pl;

    void *ws = workspace;
    if (!ws) {
        if (pl.ws_bytes > 0) {
            st = grow_library_workspace(&d->ws, &d->ws_bytes, pl.ws_bytes, true, stream);
            if (st != NORM_OK)
                return st;
        }
        ws = d->ws;
    } else if (workspace_bytes < pl.ws_bytes) {
        return NORM_ERR_WORKSPACE;
    }

    LnParams p;
    std::memset(&p, 0, sizeof(p));
    p.x = x;
    p.gamma = gamma;
    p.beta = beta;
    p.y = y;
    p.rows = rows;
    p.row_len = row_len;
    p.eps = eps;
    p.sync = static_cast<normk::LnSync *>(ws);
    p.part = ws ? reinterpret_cast<float4 *>(static_cast<char *>(ws) + kWsHeader) : nullptr;
    p.err = stream_err(*d, stream);
    p.timeout_ns = static_cast<uint64_t>(g_opt_timeout_ns.load());
    p.chunk = pl.chunk;
    p.parts = pl.parts;
    cudaError_t e;
    if (ch.ln_stream) {
        normk::GnSegParams q;
        std::memset(&q, 0, sizeof(q));
        q.x = x;
        q.gamma = gamma;
        q.beta = beta;
        q.y = y;
        q.rows = rows;
        q.seg_len = row_len;
        q.G = 1;
        q.M = row_len;
        q.S = 1;
        q.eps = eps;
        q.timeout_ns = p.timeout_ns;
        q.err = p.err;
        q.cache_gb = static_cast<size_t>(row_len) * esz <= kGbL1Bytes;
        e = normk::gns_stream_launch(q, bf16, false, ch.ln_cluster, false, stream);
    } else if (ch.row_kernel) {
        e = normk::ln_rows_launch(p, bf16, d->sm_count, stream);
    } else if (ch.persistent) {
        p.tag_skew = static_cast<unsigned>(g_opt_extra_arrivals.load());
        p.max_n4 = pl.max_n4;
        p.groups = pl.groups;
        e = normk::ln_persistent_launch(p, pl.grid, pl.dyn_smem, stream, bf16);
    } else {
        e = normk::ln_split_launch(p, bf16, pl.vec4, stream);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
    }
    return NORM_OK;
}

// RMSNorm on tensors of esz-byte elements.
norm_status_t rms_channel_fwd(const void *x, void *y, int64_t B, int64_t C, int64_t S, float eps,
                              cudaStream_t stream, int esz)
{
    int64_t bc = 0, n = 0;
    if (B < 0 || C < 0 || S < 0 || !valid_eps(eps) || !safe_mul(B, C, &bc) || !safe_mul(bc, S, &n))
        return NORM_ERR_INVALID_ARG;
    if (n == 0)
        return NORM_OK;
    if (!x || !y)
        return NORM_ERR_INVALID_ARG;
    if (!aligned(x, esz) || !aligned(y, esz))
        return NORM_ERR_MISALIGNED;
    const size_t nb = static_cast<size_t>(n) * esz;
    if (x != y && overlaps(x, nb, y, nb))
        return NORM_ERR_INVALID_ARG;
    DeviceState *d = nullptr;
    norm_status_t st = device_state(&d);
    if (st != NORM_OK)
        return st;
    if (normk::rms_channel_launch(x, y, B, C, S, eps, esz == 2, stream) != cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
    }
    return NORM_OK;
}

// GroupNorm + LeakyReLU + x2 over x[N][C][S] of esz-byte elements.  The
// (N, C) entry points pass S = 1 and nchw = false: they take the page's
// vector kernel where it applies and never the split path (they have no
// workspace).
norm_status_t group_lrelu_x2_fwd(const void *x, const void *gamma, const void *beta, void *y, int64_t N, int64_t C,
                                 int64_t S, int64_t num_groups, float eps, float negative_slope, void *workspace,
                                 size_t workspace_bytes, cudaStream_t stream, int esz, bool nchw)
{
    int64_t nc = 0, n = 0;
    if (N < 0 || C < 0 || S < 0 || num_groups <= 0 || !valid_eps(eps) || !std::isfinite(negative_slope) ||
        !safe_mul(N, C, &nc) || !safe_mul(nc, S, &n))
        return NORM_ERR_INVALID_ARG;
    if (C % num_groups != 0)
        return NORM_ERR_INVALID_ARG;
    if (n == 0)
        return NORM_OK;
    if (!x || !y)
        return NORM_ERR_INVALID_ARG;
    if (!aligned(x, esz) || !aligned(y, esz) || !aligned(gamma, esz) || !aligned(beta, esz))
        return NORM_ERR_MISALIGNED;
    const size_t nb = static_cast<size_t>(n) * esz, pb = static_cast<size_t>(C) * esz;
    if ((x != y && overlaps(x, nb, y, nb)) || overlaps(gamma, pb, y, nb) || overlaps(beta, pb, y, nb))
        return NORM_ERR_INVALID_ARG;
    if (workspace && (!aligned(workspace, 16) || overlaps(workspace, workspace_bytes, y, nb) ||
                      overlaps(workspace, workspace_bytes, x, nb)))
        return NORM_ERR_WORKSPACE;
    DeviceState *d = nullptr;
    norm_status_t st = device_state(&d);
    if (st != NORM_OK)
        return st;
    const bool bf16 = esz == 2;
    const int64_t M = C / num_groups, L = M * S, R = N * num_groups;
    const uintptr_t va = 4u * esz;
    const bool vec4 = (L & 3) == 0 && aligned(x, va) && aligned(y, va) && aligned(gamma, va) && aligned(beta, va);
    const int64_t opt = g_opt_gn_path.load();
    cudaError_t e;

    // The page's design: M a power of two in 4..128, 4 channels a thread.
    const bool pow2 = M >= 4 && M <= 128 && (M & (M - 1)) == 0;
    if (opt == 0 && S == 1 && pow2 && vec4 && (C & 3) == 0 && C / 4 < (int64_t(1) << 30)) {
        e = normk::gn_vec4_launch(x, gamma, beta, y, N, C, M, eps, negative_slope, bf16, d->sm_count, stream);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return NORM_ERR_CUDA;
        }
        return NORM_OK;
    }

    // Register path: the smallest cluster that holds a segment (or the
    // forced one), if such clusters can be resident.
    int cluster = 0;
    if (vec4) {
        const int64_t forced = g_opt_gn_cluster.load();
        const int64_t L4 = L / 4;
        cluster = forced ? static_cast<int>(forced) : gn_auto_cluster(L4);
        if (cluster && (L4 + cluster - 1) / cluster > normk::gns_reg_capacity4(1))
            cluster = 0;
        int active = 0;
        if (cluster && (normk::gns_reg_max_clusters(L, S, bf16, cluster, &active) != cudaSuccess || active < 1)) {
            cudaGetLastError();
            cluster = 0;
        }
    }
    // Streamed form of the register path: 16-byte aligned x rows and slices,
    // its own cluster size (bf16 slices hold twice as many vectors).
    bool stream_ok = false;
    int64_t stream_slice = 0;
    int stream_cl = 0;
    bool stream_wide = false;
    if (vec4 && aligned(x, 16) && (bf16 ? (L & 7) == 0 : true)) {
        const int64_t forced = g_opt_gn_cluster.load();
        const int64_t cap = normk::gns_stream_capacity4(bf16);
        stream_cl = forced ? static_cast<int>(forced) : stream_auto_cluster(L / 4, cap);
        int active = 0;
        if (stream_cl) {
            stream_slice = (L / 4 + stream_cl - 1) / stream_cl;
            stream_slice = (stream_slice + 1) & ~int64_t(1);
            stream_ok = stream_slice <= cap &&
                        normk::gns_stream_max_clusters(L, S, bf16, true, stream_cl, false, &active) == cudaSuccess &&
                        active >= 1;
        }
        if (!stream_ok)
            cudaGetLastError();
        // Groups already split over a cluster may be split over twice the
        // CTAs (half the slice each, up to clusters of 8): those CTAs hold
        // less, more of them are resident, and each cluster streams more
        // groups.  Taken when the waves of groups over the resident clusters
        // times the slice length, a model of the launch's time, is smaller.
        if (stream_ok && !forced && stream_cl >= 2) {
            const int alt = stream_auto_cluster(L / 4, cap / 2);
            int alt_active = 0;
            if (alt > stream_cl && alt <= 8) {
                if (normk::gns_stream_max_clusters(L, S, bf16, true, alt, true, &alt_active) != cudaSuccess)
                    cudaGetLastError();
            }
            if (alt_active >= 1) {
                int64_t alt_slice = (L / 4 + alt - 1) / alt;
                alt_slice = (alt_slice + 1) & ~int64_t(1);
                const int64_t waves = (R + active - 1) / active, alt_waves = (R + alt_active - 1) / alt_active;
                if (alt_waves * alt_slice < waves * stream_slice) {
                    stream_cl = alt;
                    stream_slice = alt_slice;
                    stream_wide = true;
                }
            }
        }
    }
    // Team path: segments of at most 256 items of 4, 2 or 1 elements.  The
    // automatic choice leaves its longest groups (over 128 items) to the
    // register kernel for bf16, where that kernel was measured faster.
    const bool pair = (L & 1) == 0 && aligned(x, 2u * esz) && aligned(y, 2u * esz);
    const int team_elems = vec4 ? 4 : pair ? 2 : 1;
    const int64_t team_items = L / team_elems;
    const bool team_ok = team_items <= normk::gns_team_max_items();
    const bool team_auto = team_ok && (team_items <= normk::gns_team_max_items() / 2 || !bf16 || !cluster);
    // Persistent path (the LayerNorm persistent kernel in its GroupNorm form):
    // each 16-byte unit (4 fp32 or 8 bf16 values) inside one channel (S a
    // multiple of it), 16-byte aligned x and y, x read from HBM once for
    // segments too long for a cluster to hold.
    LnPlan pp;
    const bool pers_ok = S % (16 / esz) == 0 && aligned(x, 16) && aligned(y, 16) &&
                         plan_persistent(R, L, *d, &pp, esz);
    GnPlan pl;
    if (opt == kGnPersistent && !pers_ok)
        return NORM_ERR_UNSUPPORTED;
    if (opt == kGnTeam && !team_ok)
        return NORM_ERR_UNSUPPORTED;
    if (opt == kGnReg && !cluster)
        return NORM_ERR_UNSUPPORTED;
    if (opt == kGnStream && !stream_ok)
        return NORM_ERR_UNSUPPORTED;
    if (opt == kGnSplit && !nchw)
        return NORM_ERR_UNSUPPORTED;
    if (opt)
        pl.path = static_cast<int>(opt);
    else if (team_auto)
        pl.path = kGnTeam;
    else if (stream_ok && stream_slice > kGnStreamMinPer)
        pl.path = kGnStream;
    else if (cluster)
        pl.path = kGnReg;
    else if (pers_ok && L >= kPersistentMinRowLen && nb >= kGnPersistentMinBytes)
        pl.path = kGnPersistent;
    else if (!nchw || (!vec4 && L <= kGnWarpMaxLen))
        pl.path = kGnWarp;
    else
        pl.path = kGnSplit;

    normk::GnSegParams p;
    std::memset(&p, 0, sizeof(p));
    p.x = x;
    p.gamma = gamma;
    p.beta = beta;
    p.y = y;
    p.rows = R;
    p.seg_len = L;
    p.G = num_groups;
    p.M = M;
    p.S = S;
    p.eps = eps;
    p.slope = negative_slope;
    p.timeout_ns = static_cast<uint64_t>(g_opt_timeout_ns.load());
    p.err = stream_err(*d, stream);
    p.cache_gb = S == 1 && static_cast<size_t>(L) * esz <= kGbL1Bytes;

    if (pl.path == kGnStream) {
        e = normk::gns_stream_launch(p, bf16, true, stream_cl, stream_wide, stream);
    } else if (pl.path == kGnReg) {
        e = normk::gns_reg_launch(p, bf16, cluster, stream);
    } else if (pl.path == kGnWarp) {
        e = normk::gns_warp_launch(p, bf16, d->sm_count, stream);
    } else if (pl.path == kGnTeam) {
        e = normk::gns_team_launch(p, bf16, team_elems, d->sm_count, stream);
    } else if (pl.path == kGnPersistent) {
        // Header and tagged records at the start of the workspace: the
        // library's LayerNorm workspace, or the caller's (zero-filled once;
        // the launches advance its row base and the split path never writes
        // there).
        void *ws = workspace;
        if (!ws) {
            st = grow_library_workspace(&d->ws, &d->ws_bytes, pp.ws_bytes, true, stream);
            if (st != NORM_OK)
                return st;
            ws = d->ws;
        } else if (workspace_bytes < pp.ws_bytes) {
            return NORM_ERR_WORKSPACE;
        }
        LnParams lp;
        std::memset(&lp, 0, sizeof(lp));
        lp.x = x;
        lp.gamma = gamma;
        lp.beta = beta;
        lp.y = y;
        lp.rows = R;
        lp.row_len = L;
        lp.eps = eps;
        lp.sync = static_cast<normk::LnSync *>(ws);
        lp.part = reinterpret_cast<float4 *>(static_cast<char *>(ws) + kWsHeader);
        lp.err = p.err;
        lp.timeout_ns = p.timeout_ns;
        lp.tag_skew = static_cast<unsigned>(g_opt_extra_arrivals.load());
        lp.max_n4 = pp.max_n4;
        lp.groups = pp.groups;
        normk::GnPersist gp;
        gp.G = num_groups;
        gp.M = static_cast<uint32_t>(M);
        gp.S = static_cast<uint32_t>(S);
        gp.slope = negative_slope;
        e = normk::ln_persistent_launch(lp, pp.grid, pp.dyn_smem, stream, bf16, &gp);
    } else {
        plan_gn_split(R, L, vec4, *d, &pl);
        void *ws = workspace;
        if (!ws) {
            // the partials need no initial contents
            st = grow_library_workspace(&d->gn_ws, &d->gn_ws_bytes, pl.ws_bytes, false, stream);
            if (st != NORM_OK)
                return st;
            ws = d->gn_ws;
        } else if (workspace_bytes < pl.ws_bytes) {
            return NORM_ERR_WORKSPACE;
        }
        float4 *part = reinterpret_cast<float4 *>(static_cast<char *>(ws) + gn_split_offset());
        LnParams lp;
        std::memset(&lp, 0, sizeof(lp));
        lp.x = x;
        lp.rows = R;
        lp.row_len = L;
        lp.eps = eps;
        lp.part = part;
        lp.chunk = pl.chunk;
        lp.parts = pl.parts;
        p.part = part;
        p.chunk = pl.chunk;
        p.parts = pl.parts;
        e = normk::ln_split_stats_launch(lp, bf16, pl.vec4, stream);
        if (e == cudaSuccess)
            e = normk::gns_split_apply_launch(p, bf16, pl.vec4, stream);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
    }
    return NORM_OK;
}

} // namespace

namespace normapi {

norm_status_t layer_fwd_workspace_need(const void *x, const void *gamma, const void *beta, const void *y,
                                       int64_t rows, int64_t row_len, float eps, int esz, size_t *ws_bytes)
{
    DeviceState *d = nullptr;
    LnChoice ch;
    bool empty = false;
    *ws_bytes = 0;
    const norm_status_t st = layer_plan(x, gamma, beta, y, rows, row_len, eps, nullptr, 0, esz, &d, &ch, &empty);
    if (st == NORM_OK && !empty)
        *ws_bytes = ch.pl.ws_bytes;
    return st;
}

} // namespace normapi

extern "C" {

norm_status_t norm_layer_fwd(const float *x, const float *gamma, const float *beta, float *y, int64_t rows,
                             int64_t row_len, float eps, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream)
{
    return layer_fwd(x, gamma, beta, y, rows, row_len, eps, workspace, workspace_bytes, stream, 4);
}

norm_status_t norm_layer_fwd_bf16(const uint16_t *x, const uint16_t *gamma, const uint16_t *beta, uint16_t *y,
                                  int64_t rows, int64_t row_len, float eps, void *workspace, size_t workspace_bytes,
                                  cudaStream_t stream)
{
    return layer_fwd(x, gamma, beta, y, rows, row_len, eps, workspace, workspace_bytes, stream, 2);
}

norm_status_t norm_rms_channel_fwd(const float *x, float *y, int64_t B, int64_t C, int64_t S, float eps,
                                   cudaStream_t stream)
{
    return rms_channel_fwd(x, y, B, C, S, eps, stream, 4);
}

norm_status_t norm_rms_channel_fwd_bf16(const uint16_t *x, uint16_t *y, int64_t B, int64_t C, int64_t S, float eps,
                                        cudaStream_t stream)
{
    return rms_channel_fwd(x, y, B, C, S, eps, stream, 2);
}

norm_status_t norm_group_lrelu_x2_fwd(const float *x, const float *gamma, const float *beta, float *y, int64_t N,
                                      int64_t C, int64_t num_groups, float eps, float negative_slope,
                                      cudaStream_t stream)
{
    return group_lrelu_x2_fwd(x, gamma, beta, y, N, C, 1, num_groups, eps, negative_slope, nullptr, 0, stream, 4,
                              false);
}

norm_status_t norm_group_lrelu_x2_fwd_bf16(const uint16_t *x, const uint16_t *gamma, const uint16_t *beta,
                                           uint16_t *y, int64_t N, int64_t C, int64_t num_groups, float eps,
                                           float negative_slope, cudaStream_t stream)
{
    return group_lrelu_x2_fwd(x, gamma, beta, y, N, C, 1, num_groups, eps, negative_slope, nullptr, 0, stream, 2,
                              false);
}

size_t norm_group_lrelu_x2_nchw_workspace_bytes(int64_t N, int64_t C, int64_t S, int64_t num_groups)
{
    int64_t R = 0, L = 0;
    if (N <= 0 || C <= 0 || S <= 0 || num_groups <= 0 || C % num_groups != 0 || !safe_mul(N, num_groups, &R) ||
        !safe_mul(C / num_groups, S, &L))
        return 0;
    DeviceState *d = nullptr;
    if (device_state(&d) != NORM_OK)
        return 0;
    size_t bytes = gn_split_ws_bound(R, L, *d);
    LnPlan pp;
    for (int esz = 4; esz >= 2; esz -= 2) {
        if (S % (16 / esz) == 0 && plan_persistent(R, L, *d, &pp, esz) && pp.ws_bytes > bytes)
            bytes = pp.ws_bytes;
    }
    return bytes;
}

norm_status_t norm_group_lrelu_x2_nchw_fwd(const float *x, const float *gamma, const float *beta, float *y, int64_t N,
                                           int64_t C, int64_t S, int64_t num_groups, float eps, float negative_slope,
                                           void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    return group_lrelu_x2_fwd(x, gamma, beta, y, N, C, S, num_groups, eps, negative_slope, workspace,
                              workspace_bytes, stream, 4, true);
}

norm_status_t norm_group_lrelu_x2_nchw_fwd_bf16(const uint16_t *x, const uint16_t *gamma, const uint16_t *beta,
                                                uint16_t *y, int64_t N, int64_t C, int64_t S, int64_t num_groups,
                                                float eps, float negative_slope, void *workspace,
                                                size_t workspace_bytes, cudaStream_t stream)
{
    return group_lrelu_x2_fwd(x, gamma, beta, y, N, C, S, num_groups, eps, negative_slope, workspace,
                              workspace_bytes, stream, 2, true);
}

norm_status_t norm_linear_group_lrelu_x2_fwd(const uint16_t *x, const uint16_t *w, const float *bias,
                                             const float *gamma, const float *beta, float *y, int64_t M, int64_t K,
                                             int64_t N, int64_t num_groups, float eps, float negative_slope,
                                             cudaStream_t stream)
{
    int64_t mk = 0, nk = 0, mn = 0;
    if (M < 0 || K < 0 || N < 0 || num_groups <= 0 || !valid_eps(eps) || !std::isfinite(negative_slope) ||
        !safe_mul(M, K, &mk) || !safe_mul(N, K, &nk) || !safe_mul(M, N, &mn))
        return NORM_ERR_INVALID_ARG;
    if (N % num_groups != 0)
        return NORM_ERR_INVALID_ARG;
    if (mn == 0)
        return NORM_OK;
    if (K == 0 || !x || !w || !y)
        return NORM_ERR_INVALID_ARG;
    if (!aligned(x, 2) || !aligned(w, 2) || !aligned(y, 4) || !aligned(bias, 4) || !aligned(gamma, 4) ||
        !aligned(beta, 4))
        return NORM_ERR_MISALIGNED;
    const size_t yb = static_cast<size_t>(mn) * 4, pb = static_cast<size_t>(N) * 4;
    if (overlaps(x, static_cast<size_t>(mk) * 2, y, yb) || overlaps(w, static_cast<size_t>(nk) * 2, y, yb) ||
        overlaps(bias, pb, y, yb) || overlaps(gamma, pb, y, yb) || overlaps(beta, pb, y, yb))
        return NORM_ERR_INVALID_ARG;
    // the tensor-core path: 16-byte aligned operands and rows (K % 8 == 0),
    // groups of 16, 32 or 64 channels, extents that fit its 32-bit tile
    // coordinates
    const int64_t group = N / num_groups;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || K % 8 != 0 ||
        !normk::linear_gn_group_size_ok(group) || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) ||
        K >= (int64_t(1) << 31))
        return NORM_ERR_UNSUPPORTED;
    DeviceState *d = nullptr;
    norm_status_t st = device_state(&d);
    if (st != NORM_OK)
        return st;
    normk::LinGnParams p;
    p.x = x;
    p.w = w;
    p.bias = bias;
    p.gamma = gamma;
    p.beta = beta;
    p.y = y;
    p.Mr = M;
    p.K = K;
    p.N = N;
    p.group = group;
    p.eps = eps;
    p.slope = negative_slope;
    p.timeout_ns = static_cast<uint64_t>(g_opt_timeout_ns.load());
    p.err = stream_err(*d, stream);
    if (normk::linear_gn_launch(p, d->sm_count, stream) != cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
    }
    return NORM_OK;
}

norm_status_t norm_last_error(cudaStream_t stream)
{
    DeviceState *d = nullptr;
    norm_status_t st = device_state(&d);
    if (st != NORM_OK)
        return st;
    unsigned *w = stream_err(*d, stream);
    unsigned word = 0;
    // stream-ordered: waits for this stream's work only
    if (cudaMemcpyAsync(&word, w, sizeof(word), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
    }
    if (word == 0)
        return NORM_OK;
    if (cudaMemsetAsync(w, 0, sizeof(unsigned), stream) != cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
    }
    if (word == NORM_ERR_TIMEOUT) {
        std::lock_guard<std::mutex> lock(g_mu);
        if (d->ws && cudaMemsetAsync(d->ws, 0, d->ws_bytes, stream) != cudaSuccess) {
            cudaGetLastError();
            return NORM_ERR_CUDA;
        }
    }
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
    }
    return static_cast<norm_status_t>(word);
}

} // extern "C"
