/*
 * rmsnorm.h -- C ABI of librmsnorm.so: fused RMSNorm forward and a
 * deterministic backward for NVIDIA GB300 (sm_103a).
 *
 * Operation (row i of an M x N matrix, column j):
 *   forward   rstd_i = 1 / sqrt((1/N) * sum_j x_ij^2 + eps)
 *             y_ij   = x_ij * rstd_i * w_j
 *   backward  xhat_ij = x_ij * rstd_i,  g_ij = dy_ij * w_j
 *             dx_ij   = rstd_i * (g_ij - xhat_ij * (1/N) * sum_j g_ij * xhat_ij)
 *             dw_j    = sum_i dy_ij * xhat_ij
 * Sources: "Chapter 13: Fused RMSNorm" (hello-gpu), section 13.1 equation
 * (eps inside the square root, mean over the true column count); "RMSNorm
 * backward (almost) without the column reduction", sections "The backward
 * pass", "The problem: summing across rows" and "The persistent kernel"
 * (weight gradient from per-block partial rows and a column sum, no float
 * atomics); "What a tuned RMSNorm kernel actually costs on Hopper", section
 * 05 (the backward reads the forward's fp32 reciprocal standard deviation).
 *
 * Conventions for every entry point below:
 *   - Tensors are caller-owned DEVICE memory on the current CUDA device,
 *     contiguous and row-major: x, y, dy, dx are M x N (row stride N), w is
 *     N, rstd is M, dw is N. The library keeps no pointer after a call.
 *   - `dtype` names the element types (rmsnorm_dtype_t): x, y, dy and dx
 *     share one activation type (fp32, bf16 or fp16); w has that type too,
 *     or fp32 with 16-bit activations (an fp32 master weight, "What a tuned
 *     RMSNorm kernel actually costs on Hopper", section 07). rstd and dw are
 *     always fp32. Arithmetic is fp32; each 16-bit output is rounded once,
 *     to nearest even (fp16 results beyond 65504 become infinities).
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream);
 *     results are valid once the stream has reached the call.
 *   - Return value is an rmsnorm_status_t. Arguments are checked before any
 *     CUDA call; nothing aborts or throws across this boundary.
 *     M == 0 launches no kernel and returns RMSNORM_OK (the backward then
 *     sets dw to zero, the empty sum, when dw is not NULL). M < 0, N <= 0, N > 2^31-1, an
 *     unknown dtype, a negative or NaN eps, or a NULL tensor pointer when
 *     M > 0 return RMSNORM_ERR_INVALID_ARG. rstd or dw not 4-byte aligned,
 *     or an element pointer not aligned to its element size, return
 *     RMSNORM_ERR_MISALIGNED. Pointers that are 16-byte aligned with
 *     N * element size a multiple of 16 take the vectorised kernels; any
 *     other aligned input takes a scalar kernel that gives the same results
 *     within rounding. A failed launch returns RMSNORM_ERR_CUDA.
 *   - No output may alias an input, except where an entry point says so.
 *   - Results are deterministic: the same inputs, shapes, dtype, device
 *     model and pointer-alignment class give bitwise-identical outputs,
 *     dw included (fixed reduction trees, no floating-point atomics).
 *   - The library looks up per-device state once (properties, the device
 *     status word, rmsnorm_bwd_noalloc's scratch address) and keeps it for
 *     the life of the process, in the device's primary context. Calls are
 *     not supported after cudaDeviceReset or from a non-primary context on
 *     a device the library has already used.
 */
#ifndef RMSNORM_H_
#define RMSNORM_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RMSNORM_F32 = 0,        /* x, y, dy, dx, w: fp32 */
    RMSNORM_BF16 = 1,       /* x, y, dy, dx, w: bf16 */
    RMSNORM_F16 = 2,        /* x, y, dy, dx, w: fp16 (IEEE binary16) */
    RMSNORM_BF16_W_F32 = 3, /* x, y, dy, dx: bf16; w: fp32 */
    RMSNORM_F16_W_F32 = 4   /* x, y, dy, dx: fp16; w: fp32 */
} rmsnorm_dtype_t;

typedef enum {
    RMSNORM_OK = 0,
    RMSNORM_ERR_INVALID_ARG = 1,
    RMSNORM_ERR_UNSUPPORTED = 2,
    RMSNORM_ERR_MISALIGNED = 3,
    RMSNORM_ERR_CUDA = 4,
    RMSNORM_ERR_NOMEM = 5,
    RMSNORM_ERR_DEVICE_TIMEOUT = 6,
    RMSNORM_ERR_OUT_OF_BOUNDS = 7 /* checked debug build only: a kernel access
                                     fell outside its tensor or ring and was
                                     skipped */
} rmsnorm_status_t;

/*
 * Forward. Reads x [M,N] and w [N]; writes y [M,N] and rstd [M] (fp32, the
 * per-row 1/sqrt(mean(x^2)+eps) that rmsnorm_bwd consumes).
 * One kernel launch. Source: hello-gpu chapter 13, section 13.1.
 */
int rmsnorm_fwd(const void *x, const void *w, void *y, float *rstd,
                int64_t M, int64_t N, float eps, int dtype,
                cudaStream_t stream);

/*
 * Backward. Reads x [M,N], w [N], dy [M,N] and rstd [M] (as written by
 * rmsnorm_fwd for the same x and eps; the backward takes no eps of its
 * own); writes dx [M,N] and dw [N] (fp32, overwritten, not accumulated).
 * A persistent kernel keeps each block's dw partial on chip across the rows
 * it owns and writes one partial row; a second kernel sums the partial rows
 * in a fixed order. Source: "RMSNorm backward (almost) without the column
 * reduction", section "The persistent kernel".
 * The partial rows live in a workspace that this call takes from the
 * stream-ordered allocator (cudaMallocAsync/cudaFreeAsync on `stream`);
 * RMSNORM_ERR_NOMEM if that fails. Use rmsnorm_bwd_ws to pass your own.
 * When the rows are few enough for one block (or one cluster) to take them
 * all, its partial row is dw itself: one kernel, no workspace, no allocation.
 * Up to 16 blocks' worth of rows run as one thread-block cluster whose
 * blocks add their partial rows in rank order through distributed shared
 * memory into dw: again one kernel and no workspace.
 */
int rmsnorm_bwd(const void *x, const void *w, const void *dy,
                const float *rstd, void *dx, float *dw,
                int64_t M, int64_t N, int dtype, cudaStream_t stream);

/*
 * Bytes of workspace rmsnorm_bwd_ws needs for this shape on `device`
 * (a CUDA ordinal). Returns 0 when M == 0, when one block or cluster takes
 * every row (its partial row is dw itself), or when the arguments are
 * invalid.
 */
size_t rmsnorm_bwd_workspace_size(int64_t M, int64_t N, int dtype,
                                  int device);

/*
 * rmsnorm_bwd with a caller-provided workspace: device memory of at least
 * rmsnorm_bwd_workspace_size(M, N, dtype, current device) bytes, 16-byte
 * aligned, not read by the caller until the stream reaches the end of the
 * call, and not shared with another call in flight. A smaller or NULL
 * workspace (with M > 0 and a nonzero need) returns RMSNORM_ERR_INVALID_ARG;
 * misaligned returns RMSNORM_ERR_MISALIGNED. Allocates nothing.
 */
int rmsnorm_bwd_ws(const void *x, const void *w, const void *dy,
                   const float *rstd, void *dx, float *dw,
                   int64_t M, int64_t N, int dtype,
                   void *workspace, size_t workspace_bytes,
                   cudaStream_t stream);

/*
 * Residual add fused into the forward: h = x + residual, rounded once into
 * the activation type and written to h [M,N]; then y [M,N] and rstd [M] as
 * rmsnorm_fwd computes them from that stored h (so the result equals adding
 * in the activation type and calling rmsnorm_fwd on the sum). Reads x,
 * residual (both [M,N], activation type) and w; h may be the residual or
 * the x buffer (the sum is written in place). One kernel launch. Source:
 * "Profiling, GPU utilisation and writing a fused kernel", Problem 15 (the
 * kernel takes a residual tensor, writes the sum back and normalises it;
 * the text calls this fusion the bigger win in a real model). Arguments and
 * errors as rmsnorm_fwd; residual and h follow x's rules.
 */
int rmsnorm_add_fwd(const void *x, const void *residual, const void *w,
                    void *h, void *y, float *rstd, int64_t M, int64_t N,
                    float eps, int dtype, cudaStream_t stream);

/*
 * Backward of rmsnorm_add_fwd. Reads h (the sum the forward wrote), w, dy,
 * rstd and, unless NULL, dres [M,N] (activation type): the gradient that
 * reaches h from its other uses, e.g. the next residual add. Writes
 * dx = (the norm's input gradient at h) + dres, which is the gradient of
 * both x and residual, since h = x + residual; and dw (fp32) as rmsnorm_bwd
 * does for input h. dx may be the dres buffer (accumulated in place). With
 * dres NULL this is rmsnorm_bwd on h. Workspace, arguments and errors as
 * rmsnorm_bwd; dres follows dy's rules.
 */
int rmsnorm_add_bwd(const void *h, const void *w, const void *dy,
                    const float *rstd, const void *dres, void *dx, float *dw,
                    int64_t M, int64_t N, int dtype, cudaStream_t stream);

/*
 * Size of the fixed scratch array used by rmsnorm_bwd_noalloc (16 MiB per
 * device that loads the library, held until the process exits).
 */
#define RMSNORM_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * RMSNORM_NOALLOC_SCRATCH_BYTES as the loaded library was built with it, for
 * bindings that cannot read this header's macros. Host only; no CUDA call.
 */
size_t rmsnorm_noalloc_scratch_bytes(void);

/*
 * rmsnorm_bwd for callers that cannot allocate device memory: code running
 * where cudaMalloc and the stream-ordered allocator are off limits, such as
 * under a custom allocator that owns all device memory, in a real-time loop
 * that must not allocate after start-up, or inside a runtime that forbids
 * allocator calls from library code. No counterpart on the pages: it is an
 * interface variant, same kernels and same results as rmsnorm_bwd.
 *   - Allocates nothing: the dw partial rows go to a fixed scratch array of
 *     RMSNORM_NOALLOC_SCRATCH_BYTES inside the library (one per device).
 *     Shapes whose partial rows need more (rmsnorm_bwd_workspace_size
 *     predicts the need) return RMSNORM_ERR_UNSUPPORTED and launch nothing.
 *   - The first call on each device looks up that device's scratch address
 *     (cudaGetSymbolAddress, with the device current); make that first call
 *     before capturing the stream into a CUDA graph.
 *   - Every call on a device shares the one scratch array, which keeps the
 *     last call's contents (each call rewrites every partial row it reads,
 *     so nothing needs clearing). Calls that overlap on the GPU race on it:
 *     order them, e.g. on one stream.
 *   - Arguments, outputs and other errors as rmsnorm_bwd; its bounded waits
 *     use the default one-second limit. dtype is RMSNORM_F32 or
 *     RMSNORM_BF16 only: other codes return RMSNORM_ERR_INVALID_ARG.
 */
int rmsnorm_bwd_noalloc(const void *x, const void *w, const void *dy,
                        const float *rstd, void *dx, float *dw,
                        int64_t M, int64_t N, int dtype, cudaStream_t stream);

/*
 * The naive backward, kept as an ablation to measure what the persistent
 * rmsnorm_bwd saves on the same GPU. Structure of "RMSNorm backward (almost)
 * without the column reduction", section "The naive kernel": three kernels
 * -- one block per row (one 16-byte vector per thread) recomputes rstd from
 * x and eps, writes dx and an M x N intermediate of per-element weight
 * gradient contributions dy*x*rstd rounded into the activation type; a
 * column pass sums contiguous row chunks into 64 fp32 partial rows; the
 * fixed-order column sum gives dw. About five passes over the tensor instead
 * of three, and dw carries one rounding per contribution into the
 * activation type (less accurate than rmsnorm_bwd's).
 * Reads x, w, dy [M,N]; writes dx [M,N] and dw [N] (fp32); eps as in
 * rmsnorm_fwd (no rstd input). Workspace (M*N elements plus 64*N floats)
 * from the stream-ordered allocator (RMSNORM_ERR_NOMEM if that fails).
 * Vector rows only: 16-byte aligned pointers, N * element size a multiple
 * of 16 and at most 16 KiB (one block of at most 1024 threads per row), and
 * M < 2^31; other shapes return RMSNORM_ERR_UNSUPPORTED. Other arguments and
 * errors as rmsnorm_bwd; M == 0 sets dw to zero.
 */
int rmsnorm_bwd_naive(const void *x, const void *w, const void *dy,
                      void *dx, float *dw, int64_t M, int64_t N, float eps,
                      int dtype, cudaStream_t stream);

/*
 * Device-side status. Every wait inside the kernels (on a bulk copy landing
 * in shared memory) is bounded in time; a wait that runs out records
 * RMSNORM_ERR_DEVICE_TIMEOUT in a status word on the device and the kernel
 * returns early instead of hanging. In the checked debug build (compiled
 * with RMSNORM_CHECKS) a kernel access outside its tensor, workspace or
 * shared-memory ring is skipped and recorded as RMSNORM_ERR_OUT_OF_BOUNDS.
 * This call synchronises `stream`, returns the first status recorded on the
 * current device since the last call (RMSNORM_OK if none), and clears it.
 * RMSNORM_ERR_CUDA if the synchronisation fails.
 */
int rmsnorm_get_last_device_error(cudaStream_t stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char *rmsnorm_status_string(int status);

/*
 * Time limit of each bounded wait, in nanoseconds, for kernels launched
 * after the call (process-wide; 0 restores the default of one second).
 */
void rmsnorm_set_wait_limit_ns(uint64_t ns);

/*
 * Failure-injection hook for testing the bounded waits: the next launch
 * that stages rows through bulk copies (a backward, or a forward that takes
 * the persistent ring kernel) will not issue the copy of unit `unit` (a
 * row, or a tile of rows for short rows), so the wait for it runs out and
 * the status word reads RMSNORM_ERR_DEVICE_TIMEOUT. Outputs of that call are
 * unspecified. One-shot; -1 cancels.
 */
void rmsnorm_test_drop_copy(int64_t unit);

/*
 * HBM roofline probes (the measured denominator of the throughput ratio;
 * "What a tuned RMSNorm kernel actually costs on Hopper", section 02: best
 * of a copy, a pure write and a two-read-one-write pattern). 16-byte vector
 * accesses in a grid-stride loop over `bytes` bytes (a multiple of 16; all
 * pointers 16-byte aligned):
 *   RMSNORM_PROBE_COPY   dst[k] = a[k]                      (moves 2*bytes)
 *   RMSNORM_PROBE_WRITE  dst[k] = a bit pattern of zeros     (moves bytes)
 *   RMSNORM_PROBE_2R1W   dst[k] = a[k] + b[k] as fp32       (moves 3*bytes)
 * `blocks_per_sm` (>= 1) sets the grid. Unused pointers may be NULL.
 */
typedef enum {
    RMSNORM_PROBE_COPY = 0,
    RMSNORM_PROBE_WRITE = 1,
    RMSNORM_PROBE_2R1W = 2
} rmsnorm_probe_t;

int rmsnorm_probe(int kind, void *dst, const void *a, const void *b,
                  size_t bytes, int blocks_per_sm, cudaStream_t stream);

/* Kernel family a call dispatches to. */
typedef enum {
    RMSNORM_VARIANT_NONE = 0,      /* M == 0: nothing launched */
    RMSNORM_VARIANT_ROWGROUP = 1,  /* short rows: a sub-warp or warp per row */
    RMSNORM_VARIANT_CTA_ROW = 2,   /* one thread block per row */
    RMSNORM_VARIANT_CLUSTER_ROW = 3, /* a thread-block cluster per row */
    RMSNORM_VARIANT_SCALAR = 4,    /* unaligned or ragged rows, and backward
                                      rows wider than 262144 16-bit or
                                      229376 fp32 elements */
    RMSNORM_VARIANT_TWO_PASS = 5,  /* wide rows (forward): a block per row,
                                      two passes, the second served by L2 */
    RMSNORM_VARIANT_RING = 6       /* wide rows (forward): persistent blocks
                                      (or clusters) with a ring of row slices
                                      moved by bulk copies */
} rmsnorm_variant_t;

typedef enum {
    RMSNORM_PASS_FWD = 0,     /* rmsnorm_fwd and rmsnorm_add_fwd */
    RMSNORM_PASS_BWD = 1,     /* rmsnorm_bwd, and rmsnorm_add_bwd without dres */
    RMSNORM_PASS_BWD_RES = 2, /* rmsnorm_add_bwd with dres */
    RMSNORM_PASS_FWD_ADD = 3  /* rmsnorm_add_fwd */
} rmsnorm_pass_t;

typedef struct {
    int variant;            /* rmsnorm_variant_t */
    int threads;            /* threads per block */
    int vectors_per_thread; /* 16-byte vectors of a row each thread owns */
    int threads_per_row;    /* lanes sharing one row (ROWGROUP), else threads */
    int rows_per_unit;      /* rows per block pass (row-group tile, or row
                               groups); TWO_PASS: blocks per SM */
    int cluster;            /* blocks per row (1 unless CLUSTER_ROW or RING),
                               at most 8, or 16 for backward rows over 256
                               KiB (a non-portable cluster size: on a device
                               that refuses it they run SCALAR);
                               backward ROWGROUP / CTA_ROW with cluster > 1:
                               the grid is one cluster of that many blocks,
                               which sums dw on chip (few rows) */
    int row_groups;         /* independent row groups per block (backward
                               CTA_ROW: each group of threads/row_groups
                               threads owns its own rows; else 1) */
    int stages;             /* shared-memory pipeline depth (backward) */
    int smem_bytes;         /* dynamic shared memory per block */
    int grid;               /* blocks launched; 0 when device < 0 */
    int partial_rows;       /* dw partial rows written (backward), else 0 */
    int64_t workspace_bytes;/* backward workspace: 0 for the forward, and 0
                               when one partial row (written to dw) suffices */
} rmsnorm_plan_t;

/*
 * Describe, without launching anything, what the pass named by `pass`
 * (rmsnorm_pass_t) would run for this shape with 16-byte aligned
 * pointers. With device >= 0 the grid and workspace are filled in from
 * that device's properties (needs a GPU), and a row split over a cluster
 * gets the cluster shape the calls use on that device (chosen with the
 * occupancy API, once per dtype and N); with device < 0 only the
 * width-dependent choices of the static ladder are made (host only), which
 * for such rows may differ from what runs. Returns a status code.
 */
int rmsnorm_plan(int64_t M, int64_t N, int dtype, int pass, int device,
                 rmsnorm_plan_t *out);

/* Library version as "major.minor.patch" (static storage), followed by
   "+checks" in the checked debug build. */
const char *rmsnorm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_H_ */
