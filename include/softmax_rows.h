/*
 * softmax_rows: fused, numerically stable row-wise softmax on one GB300 GPU.
 *
 * For every row i of an M x N row-major matrix x (leading dimension ld_in
 * elements), the library writes
 *
 *     y[i,j] = exp(x[i,j] - m_i) / sum_k exp(x[i,k] - m_i),  m_i = max_k x[i,k],
 *
 * to an M x N row-major matrix y (leading dimension ld_out). This is the
 * fused softmax of "Triton: Writing GPU Kernels in Python, Measured" (Step 2:
 * subtract the row maximum, exponentiate, divide by the sum, one pass over
 * the row held on chip), with the row-stride interface of "Fused Softmax on
 * GPU: From Naive PyTorch to Persistent Triton Kernels" (Triton, one block
 * per row: input and output row strides), and the numeric contract of the
 * "Warpline" README (Providers): reduction state in FP32 and a single cast
 * back to the input dtype. Wide rows use the online max/sum merge of
 * "Measured optimization case studies" (Wide rows), including its guard for
 * all -inf chunks.
 *
 * Conventions shared by every entry point:
 *   - in, out: DEVICE pointers owned by the caller; the library never frees,
 *     keeps or allocates them. The input and output dtype are the same.
 *   - M >= 0 rows, N >= 1 columns; ld_in >= N, ld_out >= N count elements.
 *     Element (i, j) is in[i*ld_in + j] / out[i*ld_out + j]. Columns
 *     [N, ld) are never read and never written.
 *   - M == 0 is a no-op returning SR_OK.
 *   - in == out with ld_in == ld_out (in place) is allowed; any other
 *     overlap is undefined.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) on the current device. Nothing blocks the
 *     host and nothing is allocated per call. The first call on a device
 *     queries and caches its properties.
 *   - Kernels are launched with programmatic stream serialisation: a call's
 *     kernel may be scheduled while the previous kernel on `stream` drains,
 *     but it waits for that kernel to complete, with its memory visible,
 *     before reading or writing any global memory. Stream order is exactly
 *     as without it; back-to-back calls overlap only their launch and block
 *     dispatch with the previous kernel's tail.
 *   - Arguments are checked before anything is launched; a rejected call
 *     launches nothing and leaves `out` untouched.
 *   - Misaligned pointers or pitches are not an error: they select plans
 *     that use narrower memory accesses.
 *   - Results follow the definition exactly in the special cases: a row that
 *     is all -inf is NaN; a NaN or +inf anywhere in a row makes the row NaN;
 *     -inf entries of an otherwise finite row give exact zeros.
 */
#ifndef SOFTMAX_ROWS_H
#define SOFTMAX_ROWS_H

#include <stdint.h>

#if defined(__GNUC__)
#define SR_API __attribute__((visibility("default")))
#else
#define SR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle type as cudaStream_t. */
typedef struct CUstream_st* sr_stream_t;

/* Element types: IEEE binary32, bfloat16 (upper half of binary32), IEEE binary16. */
enum sr_dtype { SR_F32 = 0, SR_BF16 = 1, SR_F16 = 2 };

enum sr_status {
    SR_OK = 0,
    SR_EINVAL = 1,          /* bad size, pitch or null pointer */
    SR_EDTYPE = 2,          /* unknown dtype */
    SR_ECUDA = 3,           /* a CUDA runtime call or launch failed */
    SR_EDEVICE_TIMEOUT = 4, /* a kernel's bounded wait expired (see softmax_rows_last_device_error) */
    SR_EPLAN = 5,           /* the forced plan cannot handle this shape or alignment */
    SR_EBOUNDS = 6          /* bounds-checking build: a device access fell outside the call's
                               matrices (see softmax_rows_last_device_error) */
};

/*
 * Kernel plans. AUTO picks by row width, dtype and alignment. It takes ROW
 * for rows of 256 16-byte vectors (4 KiB) up to 32 KiB (16-bit) or 64 KiB
 * (FP32), WARP for shorter rows, WIDE for wider rows, and ONLINE otherwise.
 * ROW and WIDE need rows that are aligned, or whose input and output share
 * their offset from a 16-byte boundary (WIDE: aligned only beyond 512 KiB). Every plan computes the same
 * function; forcing one (softmax_rows_ex) only changes the schedule:
 *   WARP    one warp per row, the row resident in registers; rows up to 2048 elements.
 *   CTA     one thread block per row, the row staged in shared memory by
 *           bulk asynchronous copies; aligned rows up to 32 KiB.
 *   CLUSTER one thread-block cluster per row, each block holding a slice in
 *           shared memory and the per-slice (max, sum) merged across the
 *           cluster; aligned rows up to 512 KiB. One HBM read per element.
 *   ONLINE  one thread block per row, an online (max, sum) pass over the
 *           row followed by a normalise-and-write pass; any width, any alignment.
 *   SMEM    one warp per row, each warp streaming its rows through its own
 *           ring of shared-memory slots filled by bulk asynchronous copies;
 *           no block barrier at all; aligned rows up to 32 KiB.
 *   ROW     one thread block per row loaded straight into registers, one
 *           block per row in the grid; rows up to 2048 vectors (16-bit) or
 *           4096 vectors (FP32).
 *   WIDE    one thread-block cluster per row, each block holding a slice of
 *           the row in registers, warp (max, sum) pairs merged across the
 *           cluster, the exponential recomputed for the output; rows up to
 *           512 KiB, and aligned rows of exactly 1 MiB with half of each
 *           slice in shared memory. Other wider aligned rows are streamed:
 *           each block reads its slice twice, the second time mostly from L2
 *           (on 8-block clusters through a ring of shared memory that a
 *           producer warp fills by bulk copies).
 * All plans but ROW and WIDE run a persistent grid sized to the device's SM
 * count.
 */
enum sr_plan {
    SR_PLAN_AUTO = 0,
    SR_PLAN_WARP = 1,
    SR_PLAN_CTA = 2,
    SR_PLAN_CLUSTER = 3,
    SR_PLAN_ONLINE = 4,
    SR_PLAN_SMEM = 5,
    SR_PLAN_ROW = 6,
    SR_PLAN_WIDE = 7
};

/*
 * The fused row softmax (definition above; "Triton: Writing GPU Kernels in
 * Python, Measured", Step 2, and "Fused Softmax on GPU", Triton one block per
 * row). in: M x N input at pitch ld_in; out: M x N output at pitch ld_out;
 * dtype: an sr_dtype; stream: the CUDA stream to enqueue on.
 * Returns SR_OK, or SR_EINVAL / SR_EDTYPE (nothing launched) or SR_ECUDA.
 */
SR_API int softmax_rows(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in,
                 int64_t ld_out, int dtype, sr_stream_t stream);

/*
 * softmax_rows with a forced plan (an sr_plan; SR_PLAN_AUTO behaves like
 * softmax_rows). Same arguments and results; returns SR_EPLAN, launching
 * nothing, when the plan cannot handle the shape or alignment. For tests and
 * plan sweeps ("Measured optimization case studies", Wide rows and Choosing
 * the plans from a grid: every plan forced on the same shape).
 */
SR_API int softmax_rows_ex(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in,
                    int64_t ld_out, int dtype, int plan, sr_stream_t stream);

/*
 * The plan softmax_rows would run for these arguments (an sr_plan > 0), or a
 * negative sr_status when they would be rejected. Pure host logic: launches
 * nothing and needs no device. The pointers are read only for alignment.
 */
SR_API int softmax_rows_plan(const void* in, const void* out, int64_t M, int64_t N, int64_t ld_in,
                      int64_t ld_out, int dtype);

/*
 * Host planning of a forced plan: `plan` if it can run these arguments,
 * otherwise -SR_EPLAN (or another negative status for rejected arguments).
 */
SR_API int softmax_rows_plan_check(const void* in, const void* out, int64_t M, int64_t N,
                            int64_t ld_in, int64_t ld_out, int dtype, int plan);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word, which a kernel sets when one of its bounded waits expires: a wait for
 * a bulk copy into shared memory (CTA, CLUSTER, SMEM plans) or for the
 * partial results of the other blocks of its cluster (WIDE, CLUSTER, and the
 * CLUSTER plan of the backward and the RMSNorm). Returns SR_OK,
 * SR_EDEVICE_TIMEOUT, SR_EBOUNDS (bounds-checking build only: an access was
 * refused; it takes precedence when both were recorded), or SR_ECUDA. A
 * kernel whose wait expired skips the rest
 * of its rows and returns, so the CUDA context stays usable; the output of
 * that call is then incomplete. The word is one per device, shared by every
 * stream, and the read and the clear are two steps: a kernel still running on
 * another stream can set it in between, and its report is then lost. Call
 * this when no other stream of the device has work of this library in flight,
 * or read a set word as covering all of them.
 */
SR_API int softmax_rows_last_device_error(sr_stream_t stream);

/*
 * Test hook for the bounded-wait path: runs `plan` (CTA, CLUSTER, SMEM or
 * WIDE) on the given arguments with its bulk copies, or for WIDE its
 * exchange of (max, sum) pairs, switched off, so every wait expires after
 * `timeout_ns` nanoseconds; the kernel then records SR_EDEVICE_TIMEOUT and
 * returns without writing `out`. Nothing hangs and nothing faults. Returns
 * like softmax_rows_ex.
 */
SR_API int softmax_rows_test_expiry(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in,
                             int64_t ld_out, int dtype, int plan, uint64_t timeout_ns,
                             sr_stream_t stream);

/*
 * The same softmax for matrices in HOST memory (h_in, h_out: host pointers,
 * same layout rules as softmax_rows). Rows are streamed through the device
 * in chunks: copied host -> device into the caller's device workspace
 * `d_work` (work_bytes bytes, 16-byte aligned, owned by the caller), reduced
 * there, and copied back, with copy-in, compute and copy-out of consecutive
 * chunks overlapped on three streams the library creates once per device.
 * Host buffers must be page-locked (cudaHostAlloc or cudaHostRegister) for
 * the copies to run asynchronously and overlap. The call returns once the
 * work is enqueued: `stream` waits for the whole pipeline, so synchronise it
 * before reading h_out; work queued on `stream` earlier runs first. Calls on
 * one device are enqueued one at a time (a library lock); calls that share a
 * workspace must be ordered by the caller (for example on one stream).
 * work_bytes must hold at least two staged rows; softmax_rows_host_workspace_bytes
 * gives the size for full overlap. Returns like softmax_rows, or SR_EINVAL for
 * a missing or too small workspace.
 */
SR_API int softmax_rows_host(const void* h_in, void* h_out, int64_t M, int64_t N, int64_t ld_in,
                             int64_t ld_out, int dtype, void* d_work, int64_t work_bytes,
                             sr_stream_t stream);

/*
 * Host-resident matrices read and written by the kernel itself (zero copy):
 * h_in and h_out must be page-locked host memory mapped into the device's
 * address space (cudaHostAlloc / cudaHostRegister with mapping, which is the
 * default under unified addressing) or managed memory; the kernel loads the
 * input over the host link and stores the output back, with no staging copies
 * and no workspace. Each pointer is checked with cudaPointerGetAttributes
 * before anything is launched; memory the device cannot address is refused
 * with SR_EINVAL. The host link bounds every plan here. Matrices of at
 * least 8 MiB whose rows the WIDE plan takes run on WIDE, which keeps the link
 * busiest. Other matrices get the plan softmax_rows would choose. Asynchronous on
 * `stream`: synchronise it before reading h_out. Returns like softmax_rows.
 */
SR_API int softmax_rows_host_mapped(const void* h_in, void* h_out, int64_t M, int64_t N,
                                    int64_t ld_in, int64_t ld_out, int dtype, sr_stream_t stream);

/*
 * Device workspace size (bytes) with which softmax_rows_host overlaps its
 * copies at full depth for M rows of N elements, or a negative sr_status.
 */
SR_API int64_t softmax_rows_host_workspace_bytes(int64_t M, int64_t N, int dtype);

/*
 * Masked softmax: in row i only the first L_i entries take part, the others
 * count as -inf; they are never read and are written as exact zeros. This is
 * the attention-score softmax with its mask applied in the kernel instead of
 * in the data (the -inf prefixes and masks of "Measured optimization case
 * studies", Wide rows); a row reads only its valid bytes.
 *   lengths: DEVICE array of M int32 lengths (L_i = lengths[i], clamped to
 *            [0, N]), caller-owned; or NULL.
 *   causal_period: with lengths == NULL and causal_period > 0, row i keeps
 *            L_i = min(N, i mod causal_period + 1) entries (rows holding query
 *            positions i mod causal_period of causal attention over N keys).
 *            Neither given: no mask (same as softmax_rows_ex).
 * L_i = 0, or valid entries that are all -inf, leave an all -inf row, which
 * is NaN everywhere like any all -inf row (its masked entries included).
 * plan: SR_PLAN_AUTO, SR_PLAN_WARP, SR_PLAN_ROW or SR_PLAN_ONLINE.
 * Other arguments and results as softmax_rows_ex; SR_EINVAL also for a
 * negative causal_period or for lengths and causal_period both given.
 */
SR_API int softmax_rows_masked(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in,
                               int64_t ld_out, int dtype, const int32_t* lengths,
                               int64_t causal_period, int plan, sr_stream_t stream);

/*
 * The split plan for wide rows ("Measured optimization case studies", Wide
 * rows: a row split across programs, each reducing its chunk to an online
 * (max, sum) pair, the pairs merged with the guard for all -inf chunks).
 * One cooperative kernel: its blocks form groups, each group takes one row
 * at a time, each block of a group always the same part of the row; a block
 * reduces its part and stores the pair, tagged with the step, in `workspace`;
 * two rows later it waits, bounded, for the tagged pairs of the rest of the
 * group, merges them into the row's (M, S) and reads its part again, from
 * L2, to write exp(x - M) / S. A row may span any number of SMs, so rows
 * wider than a thread-block cluster holds are read from DRAM once. Rows on
 * 16-byte boundaries are read by bulk copies into a shared-memory ring that
 * a producer warp of each block fills; other rows by each thread's own
 * loads. Before the kernel the call zeroes the slots it uses (one
 * cudaMemsetAsync on `stream`). Fastest of all entry points for FP32 rows of
 * 4 MiB and more; on narrower rows softmax_rows is as fast or faster.
 * Same arguments and layout rules as softmax_rows, plus a caller-owned
 * DEVICE workspace of at least softmax_rows_split_workspace_bytes(...) bytes
 * (a fixed size), 16-byte aligned, whose contents on entry do not matter.
 * In-place use (in == out) is rejected (SR_EINVAL): the second pass rereads
 * the input. Calls that share a workspace must not overlap on the GPU.
 * Returns like softmax_rows, or SR_EINVAL for a missing, misaligned or too
 * small workspace; an expired wait is reported by
 * softmax_rows_last_device_error (SR_EDEVICE_TIMEOUT).
 */
SR_API int softmax_rows_split(const void* in, void* out, int64_t M, int64_t N, int64_t ld_in,
                              int64_t ld_out, int dtype, void* workspace, int64_t workspace_bytes,
                              sr_stream_t stream);

/*
 * Workspace bytes softmax_rows_split needs: 262144 for every valid problem (a
 * ring of four steps of tagged (max, sum) pairs, 16 bytes each, for up to 4096
 * blocks), or a negative sr_status for invalid arguments. Pure host logic;
 * pointers are read only for alignment.
 */
SR_API int64_t softmax_rows_split_workspace_bytes(const void* in, const void* out, int64_t M,
                                                  int64_t N, int64_t ld_in, int64_t ld_out,
                                                  int dtype);

/* How softmax_rows_split cuts a problem (softmax_rows_split_shape). */
typedef struct sr_split_shape {
    int lanes;          /* groups of blocks, each taking one row at a time */
    int parts;          /* blocks per group = parts per row */
    int64_t part_units; /* units per part (the last part may be shorter) */
    int unit_elems;     /* elements per unit: 16 / element size for 16-byte
                           aligned rows, else 1 */
} sr_split_shape;

/*
 * Host query: the groups and parts softmax_rows_split would use. max_blocks:
 * how many blocks of its kernel the device holds at once; l2_bytes: the
 * device's L2 size. Either <= 0 reads it from the current device (the only
 * case that touches CUDA). Groups: as many as rows and blocks allow while
 * three rows per group fit in half the L2; parts: the blocks left per group,
 * none shorter than 256 units. Returns SR_OK and fills *shape, or an
 * sr_status (SR_EINVAL also for a null shape).
 */
SR_API int softmax_rows_split_shape(const void* in, const void* out, int64_t M, int64_t N,
                                    int64_t ld_in, int64_t ld_out, int dtype, int max_blocks,
                                    int64_t l2_bytes, sr_split_shape* shape);

/*
 * Test hook: softmax_rows_split with no block counting itself in, so that
 * every wait expires after `timeout_ns`; the call must then leave the output
 * unwritten and softmax_rows_last_device_error must report
 * SR_EDEVICE_TIMEOUT, with the context still usable.
 */
SR_API int softmax_rows_split_test_expiry(const void* in, void* out, int64_t M, int64_t N,
                                          int64_t ld_in, int64_t ld_out, int dtype,
                                          void* workspace, int64_t workspace_bytes,
                                          uint64_t timeout_ns, sr_stream_t stream);

/*
 * The split plan without a caller workspace, for callers that cannot
 * allocate device memory: code held to a fixed device-memory budget reserved
 * at start-up (inference servers, plugins inside another framework's memory
 * pool), code that must not change the device's memory footprint while it
 * runs, and code for which a cudaMalloc could implicitly synchronise the
 * device. The source pages have no counterpart; this entry point only
 * changes where the split plan keeps its statistics.
 *
 * Same arguments, results and layout rules as softmax_rows_split, without
 * the workspace: the split plan's workspace (its fixed size, every problem
 * fits) lives in an array built into the library's device image (every GPU
 * that loads the library holds it until the process exits). This call
 * allocates nothing and calls no allocating routine. The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current); make that first call before any stream capture.
 * Every call on a device shares the one array; nothing in it needs to start
 * at zero. Calls whose kernels overlap on the GPU (other streams, other host
 * threads) race on the array: order them.
 */
SR_API int softmax_rows_split_noalloc(const void* in, void* out, int64_t M, int64_t N,
                                      int64_t ld_in, int64_t ld_out, int dtype,
                                      sr_stream_t stream);

/*
 * Softmax backward ("Measured optimization case studies", Training: backward
 * kernels through autograd: the softmax keeps its output y and forms
 * y * (dy - sum(y * dy))). For every row i,
 *     dx[i,j] = y[i,j] * (dy[i,j] - sum_k y[i,k] * dy[i,k]),
 * with the sum (a dot product) held in FP32 and each dx rounded once to the
 * dtype. y, dy and dx are DEVICE M x N row-major matrices in the same dtype,
 * with pitches ld_y, ld_dy, ld_dx (elements, each >= N), caller-owned; dx
 * must not overlap y or dy (dx equal to y or dy is rejected with SR_EINVAL).
 * Pad columns [N, ld_dx) are not written. y need not be a softmax output: the
 * formula is applied as written (a NaN or infinity in a row's y or dy makes
 * that row's dot product, and so its dx, NaN or infinite).
 * Enqueued on `stream`; asynchronous like softmax_rows. Returns SR_OK,
 * SR_EDTYPE, SR_EINVAL (sizes, pitches, null pointers, aliasing, or a last
 * addressed byte beyond INT64_MAX) or SR_ECUDA.
 */
SR_API int softmax_rows_backward(const void* y, const void* dy, void* dx, int64_t M, int64_t N,
                                 int64_t ld_y, int64_t ld_dy, int64_t ld_dx, int dtype,
                                 sr_stream_t stream);

/*
 * softmax_rows_backward with a chosen plan: SR_PLAN_AUTO, SR_PLAN_ROW (a
 * team of threads per row, the row held in registers; rows up to 16384
 * elements), SR_PLAN_CLUSTER (a thread-block cluster of 2..16 blocks per row,
 * partial dot products exchanged in distributed shared memory; rows up to
 * 131072 elements held in registers, and aligned rows of any width streamed:
 * each block reads its slice once to reduce it and again to write) or
 * SR_PLAN_ONLINE (any row: y and dy are read twice). Rows are read as 16-byte
 * vectors when the three matrices' bases and pitches agree modulo 16 bytes
 * (an element-aligned head and tail are read singly); otherwise element by
 * element, and the limits halve (8192 and 65536). AUTO takes ROW for rows a
 * team of at most 256 threads holds when there are rows enough for the GPU,
 * CLUSTER for wider rows and for fewer rows than SMs, ONLINE otherwise.
 * SR_EPLAN when the plan cannot take the shape.
 */
SR_API int softmax_rows_backward_ex(const void* y, const void* dy, void* dx, int64_t M,
                                    int64_t N, int64_t ld_y, int64_t ld_dy, int64_t ld_dx,
                                    int dtype, int plan, sr_stream_t stream);

/*
 * Test hook for the bounded waits of the row-pair CLUSTER plan: runs the
 * softmax backward with SR_PLAN_CLUSTER and its partial dot products not sent,
 * so every block's wait for its peers expires after `timeout_ns` nanoseconds;
 * the kernel then records SR_EDEVICE_TIMEOUT (see softmax_rows_last_device_error)
 * and returns without writing dx. Nothing hangs and nothing faults. Returns
 * like softmax_rows_backward_ex (SR_EPLAN when the CLUSTER plan cannot take
 * the shape).
 */
SR_API int softmax_rows_backward_test_expiry(const void* y, const void* dy, void* dx, int64_t M,
                                             int64_t N, int64_t ld_y, int64_t ld_dy,
                                             int64_t ld_dx, int dtype, uint64_t timeout_ns,
                                             sr_stream_t stream);

/*
 * Host-only query: the plan softmax_rows_backward_ex would run for `plan`
 * (SR_PLAN_AUTO resolves to a concrete plan), or a negative sr_status
 * (-SR_EPLAN when the plan cannot take the shape). The pointers are only
 * inspected for alignment. sm_count > 0 stands for the device's SM count (it
 * steers the automatic choice and the cluster size); sm_count <= 0 queries
 * the current device.
 */
SR_API int softmax_rows_backward_plan(const void* y, const void* dy, const void* dx, int64_t M,
                                      int64_t N, int64_t ld_y, int64_t ld_dy, int64_t ld_dx,
                                      int dtype, int plan, int sm_count);

/*
 * Residual RMSNorm forward, the second row reduction on the same plans (the
 * "Warpline" README's K1 kernel; "Measured optimization case studies",
 * Residual RMSNorm: the input and the residual are added in FP32 and the sum
 * rounded once to the input dtype, the RMS is reduced in FP32, the weight
 * applied and the result rounded once). For every row i,
 *     h[j]   = dtype(x[i,j] + residual[i,j])
 *     y[i,j] = dtype(h[j] * weight[j] / sqrt(mean_j h[j]^2 + eps))
 * The sum h is not written anywhere. x, residual and y are DEVICE M x N
 * row-major matrices with pitches ld_x, ld_r, ld_y (elements, >= N); weight
 * is a DEVICE vector of N elements; all in the one dtype, caller-owned. y
 * must not overlap x or residual (y equal to either is rejected). eps must be
 * finite and >= 0 (eps = 0 and a zero row give NaN, 0/0). Pad columns of y
 * are not written. Plans and limits as softmax_rows_backward_ex. Returns
 * SR_OK, SR_EDTYPE, SR_EINVAL, SR_EPLAN or SR_ECUDA.
 */
SR_API int rmsnorm_residual_rows(const void* x, const void* residual, const void* weight, void* y,
                                 int64_t M, int64_t N, int64_t ld_x, int64_t ld_r, int64_t ld_y,
                                 float eps, int dtype, sr_stream_t stream);

SR_API int rmsnorm_residual_rows_ex(const void* x, const void* residual, const void* weight,
                                    void* y, int64_t M, int64_t N, int64_t ld_x, int64_t ld_r,
                                    int64_t ld_y, float eps, int dtype, int plan,
                                    sr_stream_t stream);

/* Host-only plan query for rmsnorm_residual_rows_ex, as softmax_rows_backward_plan. */
SR_API int rmsnorm_residual_rows_plan(const void* x, const void* residual, const void* weight,
                                      const void* y, int64_t M, int64_t N, int64_t ld_x,
                                      int64_t ld_r, int64_t ld_y, float eps, int dtype, int plan,
                                      int sm_count);

/* A static, human-readable name for an sr_status value. */
SR_API const char* softmax_rows_strerror(int status);

/*
 * Host-only description of how the WIDE plan runs M rows of N elements (of
 * the dtype, rows aligned or sharing their offset from a 16-byte boundary)
 * on a device with sm_count SMs: blocks per cluster (`csize`), 16-byte
 * vectors per block (`slice`), vectors each thread holds (`kv`; 0 for
 * streamed rows; 16 for aligned rows of exactly 1 MiB, of which 8 are held
 * in shared memory), and whether the rows are streamed
 * (`streamed`: each block reads its slice twice instead of holding it).
 * Any output pointer may be
 * NULL. Returns 0, or -SR_EDTYPE / -SR_EINVAL for a bad dtype or M < 0,
 * N < 1, sm_count < 1. Makes no CUDA call.
 */
SR_API int softmax_rows_wide_shape(int64_t M, int64_t N, int dtype, int sm_count, int* csize,
                                   int* kv, int64_t* slice, int* streamed);

/*
 * What the calling host thread's last kernel launch through this library
 * looked like, for result records and profiles (the pages tie kernel speed to
 * register pressure: "Measured optimization case studies", Specialize). It
 * describes the last kernel any entry point launched from this thread. Fields:
 *   registers            registers per thread of the kernel as compiled
 *   local_bytes          local memory per thread (register spills and stack)
 *   static_smem_bytes    statically declared shared memory per block
 *   dynamic_smem_bytes   dynamic shared memory the launch requested per block
 *   grid, block          blocks launched (x) and threads per block
 *   cluster              blocks per thread-block cluster (1: no cluster)
 *   name                 the kernel's symbol name, NUL-terminated (truncated)
 * The attributes come from cudaFuncGetAttributes on the current device.
 * Returns SR_OK; SR_EINVAL when info is NULL or this thread has launched no
 * kernel yet; SR_ECUDA when the attribute query fails.
 */
typedef struct sr_launch_info {
    int registers;
    int local_bytes;
    int static_smem_bytes;
    int dynamic_smem_bytes;
    int grid;
    int block;
    int cluster;
    char name[256];
} sr_launch_info;

SR_API int softmax_rows_last_launch(sr_launch_info* info);

/*
 * The copy ceiling: copies M rows of row_bytes bytes from `in` (row pitch
 * ld_in_bytes) to `out` (row pitch ld_out_bytes), both DEVICE, caller-owned,
 * not overlapping. It moves exactly the bytes a row softmax of the same shape
 * moves, with the same 16-byte streaming loads and stores (byte by byte when
 * a base, a pitch or the row length is not a multiple of 16, unless the rows
 * are co-aligned as below) and no
 * arithmetic: the measured device copy that the "Warpline" README (Ceilings)
 * takes as the roofline's bandwidth denominator, on the softmax's own shapes
 * and layouts. Rows at the same offset from a 16-byte boundary in both
 * matrices (equal base offsets and pitches modulo 16) are copied as a head,
 * 16-byte vectors and a tail. A measurement tool; no softmax entry point uses it. Bytes
 * [row_bytes, pitch) of each output row are not written. Asynchronous on
 * `stream`. Returns SR_OK, SR_EINVAL (M < 0, row_bytes < 1, a pitch below
 * row_bytes, a null pointer with M > 0, or a last byte beyond INT64_MAX;
 * nothing launched) or SR_ECUDA.
 */
SR_API int softmax_rows_copy_ceiling(const void* in, void* out, int64_t M, int64_t row_bytes,
                                     int64_t ld_in_bytes, int64_t ld_out_bytes,
                                     sr_stream_t stream);

/*
 * The two-input copy ceiling of the row-pair operations (softmax backward,
 * residual RMSNorm: two matrices read, one written): for M rows,
 * out[r][i] = a[r][i] XOR b[r][i] over row_bytes bytes, with a, b and out at
 * their own pitches (bytes), all DEVICE, caller-owned, out overlapping
 * neither input. The same bytes those operations move (their weight vector
 * aside), with 16-byte streaming loads and stores (bytes when a base, a pitch
 * or the row length is not a multiple of 16) and one XOR. A measurement tool.
 * Bytes [row_bytes, pitch) of each output row are not written. Asynchronous
 * on `stream`. Returns SR_OK, SR_EINVAL (M < 0, row_bytes < 1, a pitch below
 * row_bytes, a null pointer with M > 0, or a last byte beyond INT64_MAX;
 * nothing launched) or SR_ECUDA.
 */
SR_API int softmax_rows_copy_ceiling2(const void* a, const void* b, void* out, int64_t M,
                                      int64_t row_bytes, int64_t ld_a_bytes, int64_t ld_b_bytes,
                                      int64_t ld_out_bytes, sr_stream_t stream);

/*
 * Bounds-checking build. The library can also be built with every kernel
 * checking its own global accesses (libsoftmax_rows_check.so: the same entry
 * points, compiled with SR_BOUNDS_CHECK=1; a debug build for tests, never the
 * product). It stands in for the memory and race checkers that the "Measured
 * optimization case studies" page (CUDA reduction) runs before trusting a
 * kernel. Each kernel records the matrices of its call (inputs readable, the
 * output writable, each as rows of N valid elements at its pitch; masks,
 * weights and workspaces as runs of bytes). Every load, store and bulk copy
 * must fall inside the valid columns of one row of a matrix that allows it;
 * one that does not is skipped instead of executed (a skipped bulk copy makes
 * its bounded wait expire), and softmax_rows_last_device_error then returns
 * SR_EBOUNDS. Nothing traps.
 *
 * softmax_rows_build_flags: SR_BUILD_BOUNDS_CHECK when this is that build, else 0.
 * softmax_rows_bounds_address: the first address a check refused since the
 *   last query (then cleared); 0 when none, or in the product build.
 * softmax_rows_test_bounds_shrink: test hook of the checking build: every
 *   later kernel treats the last `bytes` bytes of each row of its writable
 *   matrices as outside, so a correct kernel's last stores must be refused
 *   (the checker's positive control; the memory itself is valid). 0 restores
 *   the exact extents. SR_EINVAL in the product build or for bytes < 0.
 */
#define SR_BUILD_BOUNDS_CHECK 1
SR_API int softmax_rows_build_flags(void);
SR_API uint64_t softmax_rows_bounds_address(void);
SR_API int softmax_rows_test_bounds_shrink(int64_t bytes);

/* Library version as major*10000 + minor*100 + patch. */
SR_API int softmax_rows_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SOFTMAX_ROWS_H */
