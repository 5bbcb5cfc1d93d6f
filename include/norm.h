/*
 * norm.h - C ABI of libnormgb300.so: fp32 reduce-then-apply normalization on
 * NVIDIA GB300 (sm_103a).
 *
 * Five operations, each one stream-ordered launch sequence of the library's
 * own CUDA kernels:
 *
 *   norm_layer_fwd                  LayerNorm over very long contiguous rows
 *   norm_rms_channel_fwd            RMSNorm over dim 1 of an NCHW tensor
 *   norm_group_lrelu_x2_fwd         per-row GroupNorm, then LeakyReLU, then x + x
 *   norm_group_lrelu_x2_nchw_fwd    the same over an NCHW tensor (groups span
 *                                   channels and positions)
 *   norm_linear_group_lrelu_x2_fwd  a Linear (tensor-core GEMM) with the
 *                                   GroupNorm + LeakyReLU + x + x in its
 *                                   epilogue
 *
 * Conventions shared by every entry point:
 *   - Pointers named x, y, gamma, beta, workspace are DEVICE pointers on the
 *     current CUDA device.  The caller owns all of them; the library never
 *     frees caller memory and allocates nothing on these calls unless a
 *     function says so (norm_layer_fwd with workspace == NULL).
 *   - Tensors are fp32, dense and contiguous in the row-major layout stated
 *     per function.  Strided (non-contiguous) views cannot be detected from a
 *     raw pointer; passing one gives wrong results, not an error.
 *   - Every call is asynchronous on `stream` (0 = the legacy default stream).
 *     Argument errors are returned synchronously, before anything is
 *     launched.  A launch failure returns NORM_ERR_CUDA.  Faults detected on
 *     the device (a grid barrier that gave up waiting) are recorded in an
 *     error word of the stream that norm_last_error(stream) reads.
 *   - y == x (exact aliasing, in place) is allowed.  Any other overlap of y
 *     with an input is rejected with NORM_ERR_INVALID_ARG.
 *   - eps must be finite and >= 0.  Sizes must be >= 0; a size of 0 in any
 *     extent makes the call a no-op that returns NORM_OK.
 *   - Pointers must be 4-byte aligned (NORM_ERR_MISALIGNED otherwise).  The
 *     fastest kernels also want 16-byte aligned pointers and extents that are
 *     multiples of 4; other valid inputs run a slower exact path.
 *   - All index arithmetic is 64-bit; tensors of more than 2^31 elements are
 *     supported.
 *
 * Thread safety: calls may be issued from several host threads.  The
 * process-wide options of norm_set_option() are read at launch time.
 */
#ifndef NORM_GB300_NORM_H
#define NORM_GB300_NORM_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NORM_OK = 0,
    NORM_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad eps, overlap, C % groups != 0 */
    NORM_ERR_MISALIGNED = 2,  /* a float pointer that is not 4-byte aligned */
    NORM_ERR_WORKSPACE = 3,   /* workspace too small or misaligned */
    NORM_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
    NORM_ERR_TIMEOUT = 5,     /* a device-side wait gave up (see norm_last_error) */
    NORM_ERR_UNSUPPORTED = 6  /* no usable device, or a request this build cannot serve */
} norm_status_t;

/* ------------------------------------------------------------------ LayerNorm
 * Defined by the LayerNorm page (POPCORNBENCH transcript "Kimi-K2.6 l1_p40",
 * opening problem analysis): for every row r of x[rows][row_len],
 *     mean_r = (1/row_len) * sum_i x[r][i]
 *     var_r  = (1/row_len) * sum_i (x[r][i] - mean_r)^2      (population)
 *     y[r][i] = (x[r][i] - mean_r) / sqrt(var_r + eps) * gamma[i] + beta[i]
 * An input of shape (B, d1, ..., dk) normalized over its last k dims is
 * rows = B, row_len = d1*...*dk.
 *
 * x, y     [rows][row_len] fp32, contiguous.
 * gamma    [row_len] elementwise weight, or NULL for weight 1.
 * beta     [row_len] elementwise bias, or NULL for bias 0.
 * workspace  device scratch of at least norm_layer_workspace_bytes(rows,
 *          row_len) bytes, 256-byte aligned, zero-filled before its first use
 *          (cudaMemset or norm_layer_workspace_reset).  The kernels keep it
 *          consistent from call to call, except after NORM_ERR_TIMEOUT, when
 *          it must be zero-filled again.  A workspace must not be shared by calls that
 *          can run at the same time (different streams).
 *          workspace == NULL: the library uses its own per-device workspace,
 *          allocated stream-ordered (cudaMallocAsync, then cudaMemsetAsync,
 *          on `stream`) the first time a call needs one or a larger one, and
 *          kept until exit; no call synchronizes the device.  Such calls must
 *          be serialized by the caller (one stream at a time, or streams
 *          ordered by events).  A call that would grow it while `stream` is
 *          being captured into a CUDA graph returns NORM_ERR_WORKSPACE: make
 *          a first call of the largest shape before capturing.
 *
 * Paths, all with a row length that is a multiple of 4 and 16-byte aligned
 * x/y/gamma/beta unless stated:
 *   - rows of at most 8,192 elements (16,384 for fp32): one launch, one
 *     CTA per row at a time, sized to the row, with the row in registers;
 *     x is read from HBM once and the workspace is not used;
 *   - longer rows of up to 131,072 elements (over less than 96 MiB of x for
 *     rows of 32,768 or more): one launch of the thread-block
 *     cluster kernel that GroupNorm over NCHW tensors uses (one group per
 *     row): each row is split over one CTA or a cluster of up to 16 CTAs,
 *     each CTA's next slices arrive by bulk copy into shared memory, and
 *     the CTAs of a row exchange their partial statistics through
 *     distributed shared memory; x is read from HBM once; no workspace;
 *   - longer rows (up to norm_layer_max_resident_row_len() fp32 elements,
 *     or twice as many bf16; a length that is a multiple of 4 fp32 or 8
 *     bf16 values and 16-byte aligned x, y, gamma and beta), and rows of
 *     32,768 elements or more when x holds 96 MiB or more: a
 *     persistent cooperative kernel (one CTA per SM) gives every CTA the
 *     same column slice of each row, holds the slice on chip (shared memory,
 *     then registers) from the moment it arrives until y is written, and
 *     merges the row's statistics across its CTAs with one bounded exchange
 *     per row; x is read from HBM once.  Rows shorter than about 3 Mi
 *     elements are spread over groups of CTAs, each group taking every k-th
 *     row, so that each row's exchange hides behind the group's next rows;
 *   - any other shape (ragged lengths, misaligned pointers), and rows of
 *     131,073 to 1,048,575 elements over less than 24 MiB of x (where its
 *     second read of x comes from L2): a two-kernel path that reads x twice.
 * All produce the same statistics definition.
 */
size_t norm_layer_workspace_bytes(int64_t rows, int64_t row_len);

norm_status_t norm_layer_fwd(const float *x, const float *gamma, const float *beta, float *y,
                             int64_t rows, int64_t row_len, float eps,
                             void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* LayerNorm on bfloat16 tensors: x, gamma, beta and y hold bfloat16 values
 * (the upper 16 bits of the fp32 encoding, passed as uint16_t); statistics and
 * arithmetic are fp32, and y is rounded to nearest even once.  This is the
 * bf16 form of the same operation; the pages work in fp32.  Same arguments,
 * workspace and errors as norm_layer_fwd, with 2-byte elements: pointers must
 * be 2-byte aligned, and the one-read paths want 8-byte aligned pointers and a
 * length that is a multiple of 4.  Paths as for fp32, except that the
 * cluster kernel and the persistent kernel want 16-byte aligned tensors and a
 * length that is a multiple of 8 (the persistent kernel keeps gamma/beta
 * packed in tensor memory and serves rows twice as long as in fp32). */
norm_status_t norm_layer_fwd_bf16(const uint16_t *x, const uint16_t *gamma, const uint16_t *beta, uint16_t *y,
                                  int64_t rows, int64_t row_len, float eps,
                                  void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* LayerNorm that allocates nothing.  The pages have no counterpart: this is a
 * service for callers that cannot allocate device memory at the time of the
 * call (inside an allocator's own callbacks, under a fixed memory pool, or
 * in a plugin that is handed only its inputs and outputs), so they can pass
 * neither a workspace nor workspace == NULL (which allocates once).
 *
 * Same operation, arguments, path choice and results as norm_layer_fwd
 * without the workspace: the scratch lives in a static device array of
 * NORM_NOALLOC_SCRATCH_BYTES (1 MiB) inside the library, held by every device
 * that loads the library until the process exits.
 *   - The row kernel and the cluster kernel use no scratch, so every shape
 *     they take is served, however many rows.  The persistent kernel uses
 *     about 20 KB.  The two-kernel path (ragged lengths, misaligned pointers)
 *     uses 256 bytes plus 16 bytes per (row, chunk).
 *   - Returns NORM_ERR_WORKSPACE, without launching, when the path chosen
 *     for the shape needs more scratch than the array holds (e.g. more than
 *     ~65,000 rows of a ragged length on the two-kernel path).
 *   - The first call on a device looks up the array's device address on the
 *     current device; make that first call before any stream capture.
 *   - A call whose path uses scratch zeroes the bytes that path uses with a
 *     stream-ordered memset, then runs the LayerNorm kernels on `stream`.
 *   - All calls on a device share the one array: calls that can overlap on
 *     the GPU (different streams, or different host threads without
 *     ordering) race and give wrong results.  Serialize them.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine. */
#define NORM_NOALLOC_SCRATCH_BYTES ((size_t)1 << 20)
norm_status_t norm_layer_fwd_noalloc(const float *x, const float *gamma, const float *beta, float *y,
                                     int64_t rows, int64_t row_len, float eps, cudaStream_t stream);

/* Zero `bytes` of a LayerNorm workspace on `stream` (stream-ordered). */
norm_status_t norm_layer_workspace_reset(void *workspace, size_t bytes, cudaStream_t stream);

/* Longest fp32 row (in elements) that the single-read persistent LayerNorm
 * kernel serves on the current device: each CTA's slice of a row must fit its
 * two shared-memory row buffers and its threads' registers (6,912 16-byte
 * units per CTA, 4,202,496 fp32 elements on a 152-SM GB300).  bf16 rows may
 * be twice as long (8 values a unit).  0 if the device cannot run the
 * kernel. */
int64_t norm_layer_max_resident_row_len(void);

/* ------------------------------------------------------------------ RMSNorm
 * Defined by the RMSNorm page (POPCORNBENCH transcript "Kimi-K2.6 l1_p36",
 * the reference model quoted in the analysis turn): for x[B][C][S] (an NCHW
 * tensor with S = H*W, or any trailing dims flattened into S),
 *     ms[b][s]   = (1/C) * sum_c x[b][c][s]^2
 *     y[b][c][s] = x[b][c][s] / sqrt(ms[b][s] + eps)
 * No affine parameters.  The channel stride is S elements.
 *
 * x, y  [B][C][S] fp32, contiguous.  Any C >= 1 and S >= 1; C <= 128 keeps a
 *       position's channels in registers (one HBM read), larger C re-reads x.
 */
norm_status_t norm_rms_channel_fwd(const float *x, float *y, int64_t B, int64_t C, int64_t S,
                                   float eps, cudaStream_t stream);

/* RMSNorm on bfloat16 x and y (uint16_t bit patterns), fp32 arithmetic, y
 * rounded to nearest even once; pointers 2-byte aligned.  Otherwise as
 * norm_rms_channel_fwd. */
norm_status_t norm_rms_channel_fwd_bf16(const uint16_t *x, uint16_t *y, int64_t B, int64_t C, int64_t S,
                                        float eps, cudaStream_t stream);

/* -------------------------------------------- GroupNorm + LeakyReLU + x + x
 * Defined by the GroupNorm page (POPCORNBENCH transcript "Kimi-K2.6 l2_p62",
 * first design turn): x[N][C] is split per row into num_groups groups of
 * M = C / num_groups CONTIGUOUS channels (group g = channels g*M .. g*M+M-1);
 *     mean, var = population mean and variance of the group's M values
 *     t  = (x - mean) / sqrt(var + eps) * gamma[c] + beta[c]
 *     l  = max(0, t) + negative_slope * min(0, t)
 *     y  = l + l
 *
 * x, y          [N][C] fp32, contiguous.
 * gamma, beta   [C] per-channel weight and bias, or NULL (1 and 0).
 * num_groups    must divide C.
 * M a power of two in 4..128 with C % 4 == 0 and 16-byte aligned pointers
 * takes the vectorized kernel (4 channels per thread).  Any other M of at
 * most 256 items (an item being 4 channels with 16-byte aligned pointers and
 * M % 4 == 0, else 2 channels with M even and 2-element aligned pointers,
 * else 1) takes a team-per-group kernel: 2^k adjacent lanes hold the group in
 * registers and reduce it with shuffles (bf16 groups over 128 items go to the
 * register kernel below).  Longer groups that are a multiple of 4 (up to
 * 131,072, 16-byte aligned pointers) take the register kernel of
 * norm_group_lrelu_x2_nchw_fwd (one CTA, or a cluster of up to 16 CTAs, per
 * group); the rest a warp-per-group kernel that re-reads the group from
 * cache.  Nothing is allocated.
 */
norm_status_t norm_group_lrelu_x2_fwd(const float *x, const float *gamma, const float *beta,
                                      float *y, int64_t N, int64_t C, int64_t num_groups,
                                      float eps, float negative_slope, cudaStream_t stream);

/* GroupNorm + LeakyReLU + x2 on bfloat16 x, gamma, beta and y (uint16_t bit
 * patterns), fp32 arithmetic, y rounded to nearest even once; pointers 2-byte
 * aligned (8-byte aligned with C % 4 == 0 for the vectorized kernel; with
 * 16-byte aligned pointers and M of 8 to 128 it takes 8 channels per thread,
 * one 16-byte access).  Otherwise as norm_group_lrelu_x2_fwd. */
norm_status_t norm_group_lrelu_x2_fwd_bf16(const uint16_t *x, const uint16_t *gamma, const uint16_t *beta,
                                           uint16_t *y, int64_t N, int64_t C, int64_t num_groups,
                                           float eps, float negative_slope, cudaStream_t stream);

/* GroupNorm + LeakyReLU + x2 over an NCHW tensor: the GroupNorm page's
 * operation (as above) where each channel has S = H*W positions.
 * x, y          [N][C][S] fp32, contiguous (NCHW with H*W flattened).
 * Group g of sample n holds channels g*M .. g*M+M-1 (M = C / num_groups) at
 * all S positions: the M*S values x[n][g*M .. g*M+M-1][0 .. S-1], which are
 * contiguous.  Their population mean and variance normalize every one of
 * them; gamma/beta [C] are per channel (or NULL: 1 and 0); then LeakyReLU
 * and x + x.  S = 1 is norm_group_lrelu_x2_fwd.
 * workspace     used only by the two-kernel and persistent paths below: at
 *               least norm_group_lrelu_x2_nchw_workspace_bytes(N, C, S,
 *               num_groups) bytes, 16-byte aligned, zero-filled once before
 *               its first use (cudaMemset or norm_layer_workspace_reset).
 *               The persistent path keeps a header and tagged records at its
 *               start, consistent from call to call; the two-kernel path
 *               writes its partials after them (from byte 10,496), so any
 *               mix of calls may share it as long as they are serialized
 *               (one stream).  After a NORM_ERR_TIMEOUT it must be
 *               zero-filled again.  NULL: the library allocates its own,
 *               stream-ordered (cudaMallocAsync on `stream`), on first need
 *               and keeps it (such calls must be serialized by the caller;
 *               growth during a stream capture returns NORM_ERR_WORKSPACE);
 *               the persistent path then shares the library's LayerNorm
 *               workspace.  It must not be a LayerNorm workspace that is
 *               still in use.
 * Paths (L = M*S):
 *   - groups of at most 256 items (4, 2 or 1 elements an item, as for
 *     norm_group_lrelu_x2_fwd): one launch, a team of adjacent lanes per
 *     group, statistics by shuffles, x read once;
 *   - L a multiple of 4 with 16-byte aligned pointers and L <= 131,072: one
 *     launch; each group is held in registers by one CTA or by a thread-
 *     block cluster of up to 16 CTAs that reduce the statistics through
 *     distributed shared memory; x is read from HBM once.  Where each CTA's
 *     share of a group is 1,024 elements or more (and, for bf16, L is a
 *     multiple of 8), a persistent grid of clusters streams the next group
 *     into shared memory by bulk copy while the current one is reduced (a
 *     group already split over a cluster may be split over twice the CTAs,
 *     up to 8, when the waves of groups over the resident clusters make
 *     that faster);
 *     its waits are bounded by NORM_OPT_BARRIER_TIMEOUT_NS (a CTA that gives
 *     up records NORM_ERR_TIMEOUT and leaves its part of the remaining
 *     groups of y unwritten);
 *   - groups of more than 131,072 values with S a multiple of 4 (fp32) or 8
 *     (bf16) and 16-byte aligned x and y, up to
 *     norm_layer_max_resident_row_len() values (twice that in bf16), x of
 *     48 MiB or more (smaller x is re-read mostly from L2 by
 *     the two-kernel path, which is then faster): the persistent LayerNorm
 *     kernel in its GroupNorm form (one
 *     launch, x read from HBM once; each segment is split over the CTAs of
 *     a row group, which exchange partial statistics through the workspace;
 *     gamma/beta are read per channel; waits bounded as for
 *     norm_layer_fwd, a timeout leaves y partly unwritten);
 *   - other long groups and unaligned vectors: a statistics kernel writes
 *     per-chunk partials to the workspace and an apply kernel re-reads x;
 *   - non-vector groups of 257 to 4,096 elements: one warp per group.
 */
size_t norm_group_lrelu_x2_nchw_workspace_bytes(int64_t N, int64_t C, int64_t S, int64_t num_groups);

norm_status_t norm_group_lrelu_x2_nchw_fwd(const float *x, const float *gamma, const float *beta, float *y,
                                           int64_t N, int64_t C, int64_t S, int64_t num_groups, float eps,
                                           float negative_slope, void *workspace, size_t workspace_bytes,
                                           cudaStream_t stream);

/* The bfloat16 form (uint16_t bit patterns, fp32 arithmetic, y rounded to
 * nearest even once; pointers 2-byte aligned, 8-byte aligned for the vector
 * paths).  Otherwise as norm_group_lrelu_x2_nchw_fwd. */
norm_status_t norm_group_lrelu_x2_nchw_fwd_bf16(const uint16_t *x, const uint16_t *gamma, const uint16_t *beta,
                                                uint16_t *y, int64_t N, int64_t C, int64_t S, int64_t num_groups,
                                                float eps, float negative_slope, void *workspace,
                                                size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------- Linear + GroupNorm + LeakyReLU + x + x
 * The GroupNorm page's whole module (POPCORNBENCH transcript "Kimi-K2.6
 * l2_p62": forward = F.linear(x, W, bias), then GroupNorm + LeakyReLU + x + x
 * as in norm_group_lrelu_x2_fwd; the page's first design turn weighs
 * computing the group statistics in the GEMM's epilogue), in one kernel:
 *     h[m][n] = sum_k x[m][k] * W[n][k] + bias[n]
 *     y[m][.] = norm_group_lrelu_x2 of the row h[m][.] (groups of N/num_groups
 *               contiguous channels, gamma/beta per channel)
 * h is never written to memory: the group statistics are taken in the
 * epilogue of the tensor-core GEMM, from its fp32 accumulators.
 *
 * x        [M][K] bfloat16 (uint16_t bit patterns), contiguous.
 * W        [N][K] bfloat16, contiguous: one row per output channel, the layout
 *          nn.Linear stores its weight in.
 * bias, gamma, beta  [N] fp32, or NULL (0, 1 and 0).
 * y        [M][N] fp32, contiguous; must not overlap any input.
 * Products are exact in fp32 and accumulated in fp32 by the tensor cores (in
 * an order of their own); the epilogue is fp32 (two-pass group statistics).
 * This is a bfloat16-input form: the pages' fp32 Linear is not reproduced
 * bit for bit, and results match a float64 evaluation on the same bfloat16
 * values within 1e-4 (1 + |y|).
 * Requirements (NORM_ERR_UNSUPPORTED otherwise): x, W and y 16-byte aligned,
 * K a multiple of 8, N / num_groups one of 16, 32 or 64, and M, N, K below
 * 2^31.  Any M and N (multiples of the group size) are served; rows and
 * channels past a 128 x 256 tile edge are masked.  Nothing is allocated.
 * Waits inside the kernel are bounded by NORM_OPT_BARRIER_TIMEOUT_NS (a
 * timeout is reported by norm_last_error on the stream).
 */
norm_status_t norm_linear_group_lrelu_x2_fwd(const uint16_t *x, const uint16_t *w, const float *bias,
                                             const float *gamma, const float *beta, float *y, int64_t M, int64_t K,
                                             int64_t N, int64_t num_groups, float eps, float negative_slope,
                                             cudaStream_t stream);

/* ------------------------------------------------------------------ status
 * Every stream has its own error word on each device (the first 255 streams
 * a device sees; further streams share one word).  A launch records its
 * first device-side failure in the word of the stream it was launched on
 * (for a CUDA graph: the stream it was captured on).
 * norm_last_error(stream) synchronizes `stream` only, then reads and clears
 * that stream's word.  Returns NORM_OK if no device-side wait of a call on
 * this stream gave up since the last call, else the recorded status
 * (NORM_ERR_TIMEOUT).  After a timeout the library-owned LayerNorm workspace
 * of this device is reset here (stream-ordered on `stream`);
 * caller-owned workspaces must be reset by the caller.  Returns
 * NORM_ERR_CUDA if the synchronize itself fails.
 */
norm_status_t norm_last_error(cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char *norm_status_string(norm_status_t status);

/* ------------------------------------------------------------------ options
 * Process-wide knobs, read when a call launches.  Not meant to be changed
 * while other threads are launching.
 *   NORM_OPT_LN_PATH             0 = choose automatically, 1 = force the
 *                                persistent single-read kernel, 2 = force the
 *                                two-kernel path, 3 = force the row kernel,
 *                                4 = force the thread-block cluster kernel
 *                                (1, 3 and 4: error NORM_ERR_UNSUPPORTED if
 *                                the shape does not fit).
 *   NORM_OPT_BARRIER_TIMEOUT_NS  how long a CTA waits at the LayerNorm grid
 *                                barrier (or for its own bulk copies) before
 *                                it records NORM_ERR_TIMEOUT and stops.  CTAs
 *                                stop independently: after a timeout every
 *                                element of y either keeps its previous value
 *                                or holds its correct result.  Default 200 ms;
 *                                waits that drain a CTA's own copies before it
 *                                exits use at least 100 ms.  A limit below 1 us
 *                                makes every wait for a CTA's own bulk copy
 *                                that is not over at its first (non-blocking)
 *                                look give up at once.
 *   NORM_OPT_BARRIER_EXTRA_ARRIVALS  test hook: when > 0, the grid barrier
 *                                waits for partial statistics that no CTA
 *                                publishes, so it can only end by timing
 *                                out.  Default 0.
 *   NORM_OPT_LN_CTAS             CTAs of the persistent kernel (0 = one per
 *                                SM, the default).
 *   NORM_OPT_GN_PATH             GroupNorm: 0 = choose automatically, 1 =
 *                                force the register kernel, 2 = force the
 *                                two-kernel path (NCHW entry points only),
 *                                3 = force the warp-per-group kernel, 4 =
 *                                force the streamed register kernel, 5 =
 *                                force the team-per-group kernel (groups of
 *                                at most 256 four-element vectors, or 256
 *                                elements when the vector form is off), 6 =
 *                                force the persistent single-read kernel (NCHW
 *                                with S a multiple of 4 fp32 or 8 bf16 values)
 *                                (error NORM_ERR_UNSUPPORTED where the forced
 *                                path cannot serve the call).
 *   NORM_OPT_GN_CLUSTER          CTAs per group of the register kernel: 0 =
 *                                the fewest that hold a group, or 1, 2, 4, 8
 *                                or 16.
 * Returns NORM_ERR_INVALID_ARG for an unknown option or a negative value.
 */
typedef enum {
    NORM_OPT_LN_PATH = 1,
    NORM_OPT_BARRIER_TIMEOUT_NS = 2,
    NORM_OPT_BARRIER_EXTRA_ARRIVALS = 3,
    NORM_OPT_LN_CTAS = 4,
    NORM_OPT_GN_PATH = 5,
    NORM_OPT_GN_CLUSTER = 6
} norm_option_t;

norm_status_t norm_set_option(norm_option_t option, int64_t value);
int64_t norm_get_option(norm_option_t option);

#ifdef __cplusplus
}
#endif

#endif /* NORM_GB300_NORM_H */
