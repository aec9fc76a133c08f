/*
 * mbrs_softmax.h -- C ABI of the GB300 (sm_103a) fused row softmax.
 *
 * The operation (page "Dissecting Memory Bandwidth & SRAM Tiling in Triton:
 * From GEMM to FlashAttention-3", section "The Mathematical Remedy: Online
 * Softmax Tiling"; page "I Wrote My First GPU Kernel", section "What Fusion
 * Actually Does"):
 *
 *     y[r, c] = exp(x[r, c] - m_r) / sum_k exp(x[r, k] - m_r),  m_r = max_k x[r, k]
 *
 * for every row r < rows and column c < cols, each element read from memory
 * once and written once (page "fused-softmax-roofline": one read and one
 * write per element; page "Kernel Fusion": 128 MB instead of 512 MB for a
 * 4096 x 4096 fp32 matrix).
 *
 * Layout (page "GPU Kernels - Implementing and optimizing Softmax", section
 * "Baseline & Triton Softmax kernel": rows addressed as base + row * stride):
 *   - row-major; element (r, c) of `in` is at in + r * row_stride + c and the
 *     result goes to out + r * row_stride + c (strides in ELEMENTS, one stride
 *     for both buffers, row_stride >= cols);
 *   - in and out hold the same dtype: IEEE binary32, binary16 or bfloat16;
 *   - columns cols .. row_stride-1 of each row are never written and never
 *     affect the result (they may hold anything; for 16-bit types the
 *     aligned 16-byte vectors that hold a row's first and last element are
 *     loaded whole and the elements outside the row discarded);
 *   - arithmetic is fp32 (one exp per element); the result is rounded once
 *     to the output dtype, round-to-nearest-even.
 *
 * Values: -inf entries are masked entries (they get 0).  A row with no finite
 * max -- every entry -inf -- or with a NaN or +inf entry comes out all NaN.
 *
 * Ownership: the caller owns both device buffers and the stream.  `out` is
 * never pre-initialised (page "I Wrote My First GPU Kernel", section "The
 * Honest Part": empty_like instead of zeros_like).  in == out (exact
 * aliasing) is allowed; any other overlap of the two byte ranges is rejected.
 * The library allocates no device memory per call: every path keeps its
 * partial (max, sum) states on chip (registers, shared memory, or the
 * distributed shared memory of a thread-block cluster), except path 8 (out
 * != in only), which keeps them in the output rows before it overwrites them.  Calls are
 * asynchronous on `stream`; nothing is synchronised.
 *
 * Errors: arguments are checked on the host before any launch and a status
 * code is returned (no launch happens unless the status is SOFTMAX_OK).
 * Asynchronous device faults surface at the caller's next synchronisation as
 * with any CUDA library.  Bounded waits inside the kernels that run out set a
 * device error word; softmax_check_device_error() reads it.
 */
#ifndef MBRS_SOFTMAX_H
#define MBRS_SOFTMAX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream handle, declared here when its headers are absent. */
#if !defined(__DRIVER_TYPES_H__)
struct CUstream_st;
typedef struct CUstream_st *cudaStream_t;
#endif

typedef enum {
    SOFTMAX_F32 = 0,  /* IEEE binary32 */
    SOFTMAX_F16 = 1,  /* IEEE binary16 */
    SOFTMAX_BF16 = 2  /* bfloat16 (top half of a binary32) */
} softmax_dtype_t;

typedef enum {
    SOFTMAX_OK = 0,
    SOFTMAX_ERR_NULL = 1,        /* in or out is NULL while rows > 0 */
    SOFTMAX_ERR_SHAPE = 2,       /* rows < 0, cols < 1, or the extent overflows int64 */
    SOFTMAX_ERR_STRIDE = 3,      /* row_stride < cols */
    SOFTMAX_ERR_DTYPE = 4,       /* dtype not a softmax_dtype_t */
    SOFTMAX_ERR_OVERLAP = 5,     /* in and out overlap without being equal */
    SOFTMAX_ERR_UNSUPPORTED = 6, /* a forced path that cannot take this shape */
    SOFTMAX_ERR_CUDA = 7,        /* a CUDA runtime call or launch failed */
    SOFTMAX_ERR_TIMEOUT = 8,     /* a bounded device wait ran out (device error word) */
    SOFTMAX_ERR_ALIGN = 9,       /* in or out not aligned to its element size */
    SOFTMAX_ERR_ARG = 10,        /* a bad argument to a diagnostic call */
    SOFTMAX_ERR_SCRATCH_LIMIT = 11 /* softmax_fwd_noalloc: rows exceed its fixed scratch array */
} softmax_status_t;

/* Kernel paths the dispatcher chooses between.  (5 is unused: it named a
 * TMA-fed ring of shared-memory stages, measured slower than paths 2 and 6 at
 * every width and removed; forcing it returns SOFTMAX_ERR_ARG.) */
typedef enum {
    SOFTMAX_PATH_AUTO = 0,    /* width-based choice (default) */
    SOFTMAX_PATH_WARP = 1,    /* a warp (or 2..16 lanes) per row */
    SOFTMAX_PATH_CTA = 2,     /* a thread block per row, row held in registers (any alignment) */
    SOFTMAX_PATH_CLUSTER = 3, /* 16-bit rows: a thread-block cluster per row, each block holding
                                 its slice in registers, (max, sum) exchanged through distributed
                                 shared memory */
    SOFTMAX_PATH_SPLIT = 4,   /* softmax_fwd_noalloc only: rows split across the whole grid, pass 1
                                 writes per-chunk (max, sum) into the library's fixed array, pass 2
                                 merges them, re-reads and writes.  softmax_fwd never takes it
                                 (forcing it returns SOFTMAX_ERR_ARG) */
    SOFTMAX_PATH_STREAM = 6,  /* a cluster (<= 16 blocks) per row, each block streaming its slice
                                 of any length twice: pass 1 (max, sum), exchange through
                                 distributed shared memory, pass 2 re-read and write; no scratch */
    SOFTMAX_PATH_PACKED = 7,  /* narrow rows of a dense matrix (row_stride == cols) staged through
                                 shared memory many rows at a time as one contiguous span of
                                 whole 16-byte vectors; one thread per row */
    SOFTMAX_PATH_GRID = 8     /* a few very long rows (rows * 16 < SMs, rows of 1 MiB or more) when
                                 out != in: each row cut into chunks over the whole grid, in two
                                 launches -- each chunk's (max, sum) written into a state region
                                 at the start of its output row (8 bytes per chunk and a 32-bit
                                 counter), then every block folds its row's states, re-reads its
                                 chunk and writes it, the region's own outputs written by the
                                 block of the row that counts itself last; nothing allocated.  The
                                 counter is an atomic add on `out`: host memory takes it only
                                 where the device performs atomics on host memory natively
                                 (otherwise the automatic choice is path 6) */
} softmax_path_t;

/*
 * softmax_fwd -- the fused row softmax described above.
 *   in, out     element-aligned pointers to memory the device addresses
 *               directly: device memory, or host memory that is page-locked
 *               and mapped (cudaHostAlloc, cudaHostRegister), or pageable host
 *               memory on a device that reaches it through the host's page
 *               tables (a coherent CPU-GPU link); may be NULL only if rows == 0
 *   rows        number of rows (>= 0); rows == 0 returns SOFTMAX_OK and launches nothing
 *   cols        valid columns per row (>= 1)
 *   row_stride  distance between row starts in elements (>= cols), both buffers
 *   dtype       a softmax_dtype_t
 *   stream      the CUDA stream to launch on (0 = legacy default stream)
 * Rows too long for the registers of a block or cluster (path 6) are read
 * twice, the second read usually served by L2: 3 element crossings instead of
 * 2, and still no scratch.  Allocates nothing.  Returns a softmax_status_t.
 */
int softmax_fwd(const void *in, void *out, int64_t rows, int64_t cols, int64_t row_stride,
                int dtype, cudaStream_t stream);
/* (Path 8 uses the caller's `out` rows as the place where partial states
 * meet before it overwrites them with the results; what `out` holds before
 * the call never matters, as on every path.) */

/*
 * softmax_fwd_masked -- the row softmax of scaled, causally masked scores.
 * (Page "Dissecting Memory Bandwidth & SRAM Tiling in Triton: From GEMM to
 * FlashAttention-3", section "Writing the Kernel in OpenAI Triton": the score
 * row is multiplied by the scale, and key j of query i is kept only when
 * j <= i, the others becoming -inf before the softmax.)
 * Row r is query q = r mod rows_per_seq of its group of rows (rows_per_seq
 * == 0: q = r) and keeps the columns c <= q + causal_offset:
 *     y[r,c] = exp(s_c - m) / sum over kept k of exp(s_k - m),
 *     s_c = scale * x[r,c],  m = the max of the kept s,
 * and y[r,c] = 0 for the masked columns.  Masked entries of `in` never
 * affect the result (they may hold anything; only the 16-byte vector holding
 * a row's last kept entry is loaded past it, and discarded); every column of
 * `out` is written.  A row
 * that keeps no column, or has a NaN or +inf among its kept entries, comes
 * out all NaN.
 *   scale          finite and > 0 (else SOFTMAX_ERR_ARG)
 *   causal_offset  any value; <= -1 - q masks all of query q's row
 *   rows_per_seq   >= 0 (else SOFTMAX_ERR_ARG)
 * The other arguments, the layout, aliasing and status codes are those of
 * softmax_fwd.  Runs the warp and block shapes of paths 1 and 2, or the
 * streaming cluster (path 6) for longer rows; allocates nothing; ignores the
 * autotune cache (softmax_set_force_path applies, other forced paths map to
 * path 6).
 */
int softmax_fwd_masked(const void *in, void *out, int64_t rows, int64_t cols, int64_t row_stride,
                       int dtype, float scale, int64_t causal_offset, int64_t rows_per_seq,
                       cudaStream_t stream);

/*
 * softmax_masked_copy -- a diagnostic: the memory traffic of the matching
 * softmax_fwd_masked call with no arithmetic.  Each row's kept columns (the
 * same rule: c <= (r mod rows_per_seq) + causal_offset) are copied from in to
 * out bit for bit and its other columns are set to zero bits, one block of
 * `threads` threads per row (0 = 256; else a power of two from 32 to 1024).
 * Timed beside softmax_fwd_masked it gives the time the masked call's access
 * pattern takes on its own, as a same-bytes device-to-device copy does for
 * softmax_fwd.  Rows of whole 16-byte vectors only (in and out 16-byte
 * aligned, row_stride and cols multiples of 16 bytes; else
 * SOFTMAX_ERR_UNSUPPORTED); other arguments and status codes as
 * softmax_fwd_masked.  Allocates nothing.
 */
int softmax_masked_copy(const void *in, void *out, int64_t rows, int64_t cols, int64_t row_stride, int dtype,
                        int64_t causal_offset, int64_t rows_per_seq, int threads, cudaStream_t stream);

/*
 * softmax_fwd_host -- the same softmax for a matrix in host memory, written
 * back to host memory.  (The pages have no counterpart: they time device
 * buffers only; this is the call whose end-to-end throughput includes the
 * host <-> device copies.)
 *   in_host, out_host  host pointers (may be equal); page-locked memory lets the
 *                      copies run asynchronously and overlap, pageable memory
 *                      works but the driver then stages and serialises them
 *   workspace          device memory the caller owns (256-byte aligned),
 *                      workspace_bytes long: three slots of at least one row
 *                      each; softmax_host_workspace_bytes(rows, cols,
 *                      row_stride, dtype, 0) gives the recommended size.
 *                      workspace == NULL with workspace_bytes == 0 selects
 *                      the zero-copy mode: the kernels read in_host and write
 *                      out_host in place, each element crossing the CPU-GPU
 *                      link once in each direction inside them.  Both ranges
 *                      must be memory the device reaches at the same address
 *                      (page-locked and mapped, or pageable on a device that
 *                      uses the host's page tables, as over NVLink-C2C); the
 *                      call checks the first and last byte of each range and
 *                      returns SOFTMAX_ERR_ARG without launching otherwise
 *   stream             the call is ordered after the work already queued on
 *                      stream, and work queued on stream afterwards waits for
 *                      it; it returns without waiting (synchronise stream
 *                      before reading out_host)
 * The rows move in chunks through the three workspace slots on three streams
 * of the library's own, so that the host-to-device copy of one chunk, the
 * softmax of another and the device-to-host copy of a third are in flight at
 * once.  Only the rows' cols elements are copied (pitched copies): padding
 * between host rows is neither read nor written.  Calls on one device are serialised by a lock while they are queued.
 * In the zero-copy mode the call is softmax_fwd on the host pointers (one
 * kernel, same paths and ordering on `stream`).  Other arguments, layout,
 * aliasing and status codes as softmax_fwd (SOFTMAX_ERR_ARG for a workspace
 * too small).  Allocates nothing on the device; the streams and events are
 * created once per device.
 */
int softmax_fwd_host(const void *in_host, void *out_host, int64_t rows, int64_t cols, int64_t row_stride,
                     int dtype, void *workspace, int64_t workspace_bytes, cudaStream_t stream);

/*
 * Workspace for softmax_fwd_host: three chunks of about chunk_bytes of row
 * data each (<= 0: a quarter of the matrix, within 2 to 8 MiB), whole rows
 * packed densely, never more than the matrix needs.  softmax_fwd_host makes
 * its chunks as large as the workspace it is given allows, so the workspace
 * size sets the pipeline's granularity.  Returns the
 * bytes, or a negated softmax_status_t on bad arguments.
 */
int64_t softmax_host_workspace_bytes(int64_t rows, int64_t cols, int64_t row_stride, int dtype,
                                     int64_t chunk_bytes);

/* A static English string for a status code (never NULL). */
const char *softmax_status_string(int status);

/* The path (softmax_path_t) that the last successful softmax_fwd on any thread took. */
int softmax_last_path(void);

/*
 * Test and tuning hook: force every following call onto `path` (0 = automatic).
 * threads / vpt / group override the launch shape where > 0 (threads per block,
 * 16-byte vectors per thread, and lanes per row / cluster size for paths 1 /
 * 3 and 6; for path 7 vpt is the rows each thread takes per staged span and
 * group must be 0 or 1; for path 8 group is the chunks per row, and threads x
 * vpt one of 256 x 4, 256 x 8, 512 x 4, 1024 x 4).  A forced
 * shape that cannot cover the row, or path 8 with in == out, makes
 * softmax_fwd return SOFTMAX_ERR_UNSUPPORTED.  Paths 4 and 5, and values
 * outside 0..8, return SOFTMAX_ERR_ARG and leave the setting unchanged.
 * Process-wide, not thread-safe.
 */
int softmax_set_force_path(int path, int threads, int vpt, int group);

/* Description of the launch softmax_fwd would make (host only, no GPU work). */
typedef struct {
    int path;              /* softmax_path_t actually chosen */
    int threads;           /* threads per block */
    int vpt;               /* 16-byte vectors per thread per tile (7: rows per lane group per span) */
    int group;             /* lanes per row (1), cluster size (3, 6), chunks per row (8), else 1 */
    int launches;          /* kernels per call (1; 2 for path 8) */
    int vec_store;         /* 1 if out has in's 16-byte phase (vector stores) */
    int64_t grid;          /* blocks of the kernel */
    int64_t smem_bytes;    /* dynamic shared memory per block */
    int64_t scratch_bytes; /* device scratch the call needs: 0 on every path */
    int64_t hbm_bytes;     /* bytes moved: 2 * rows * cols * elem (3x for STREAM and GRID,
                              whose second read is usually served by L2) */
    int whole_vectors;     /* 1 if every row is whole 16-byte vectors (in and out 16-byte
                              aligned, row stride and width multiples of 16 bytes): the
                              kernels then run their variants without edge tests */
} softmax_plan_t;

/*
 * softmax_plan -- fill *plan with the launch softmax_fwd would make for these
 * arguments (pointer alignment given by in_addr / out_addr, which are only
 * inspected, never dereferenced).  num_sms > 0 plans for a GPU with that many
 * SMs without touching CUDA; num_sms == 0 queries the current device.
 * Honours softmax_set_force_path.  Returns a softmax_status_t.
 */
int softmax_plan(uint64_t in_addr, uint64_t out_addr, int64_t rows, int64_t cols,
                 int64_t row_stride, int dtype, int num_sms, softmax_plan_t *plan);

/*
 * Synchronise `stream`, then read and clear this device's error word.
 * Returns SOFTMAX_ERR_TIMEOUT if a bounded wait ran out in any kernel since the
 * last check, SOFTMAX_ERR_CUDA if the synchronisation failed or a cluster
 * kernel found itself launched without clusters (it then did nothing), else
 * SOFTMAX_OK.
 */
int softmax_check_device_error(cudaStream_t stream);

/*
 * Test hooks for the bounded waits of the cluster paths (CLUSTER, STREAM and
 * the masked STREAM).  wait_limit_ns bounds each wait for the cluster's
 * (max, sum) exchange (default 1 s; <= 0 restores it; values above 1 s are
 * capped at 1 s, since the waits time 32-bit intervals).  starve != 0 makes
 * the next launches send no state, so every exchange wait can only run out:
 * the kernel records SOFTMAX_ERR_TIMEOUT, skips its stores and returns
 * normally.  Process-wide, not thread-safe.
 */
int softmax_set_wait_test(int64_t wait_limit_ns, int starve);

/*
 * Launch overlap (programmatic dependent launch), on by default.  With
 * enable != 0 each kernel this library launches may be scheduled while the
 * previous kernel in its stream is still finishing; before it reads or writes
 * any global memory it waits on the device (griddepcontrol.wait) until that
 * kernel has completed and its writes are visible, so the results are the
 * same either way.  What overlaps is the launch latency and block placement,
 * most visible for small inputs and for calls issued back to back.
 * enable == 0 launches in plain stream order.  Process-wide; returns
 * SOFTMAX_OK.
 */
int softmax_set_launch_overlap(int enable);

/*
 * softmax_fwd_noalloc -- the grid-wide split path for callers that cannot
 * allocate device memory.  (The pages have no counterpart: this entry point
 * answers a deployment constraint, not a step of the method.)
 *
 * The split path cuts every row into chunks spread over all SMs, which suits
 * a few very long rows.  Its two passes meet in a global array of per-chunk
 * (s, l) states: scratch memory.  (softmax_fwd spreads such rows the same way
 * without scratch when out != in, keeping the states in the output rows: path
 * 8; in place it can give a row at most 16 SMs, path 6 -- one fp32 row of
 * 4 M elements: 11.1 us here against 34.8 us.)  Some callers cannot obtain scratch: code running under an
 * allocator that a host framework owns exclusively, real-time loops where an
 * allocation's latency or failure is not acceptable, or processes that must
 * not grow their device footprint after start-up.  This entry point keeps the
 * states in a fixed array of SOFTMAX_NOALLOC_MAX_STATES (s, l) pairs
 * (512 KiB) compiled into the library; every GPU that loads the library holds
 * that array until the process exits.  It calls no cudaMalloc, cudaFree or
 * other allocating routine.  It always takes the split path (two passes, 3
 * element crossings).
 *   - Arguments, layout and status codes are those of softmax_fwd.  rows may
 *     be at most SOFTMAX_NOALLOC_MAX_STATES; larger calls return
 *     SOFTMAX_ERR_SCRATCH_LIMIT before any launch (each row needs at least one
 *     state; chunks per row are reduced to fit).
 *   - Every call looks up the array's device address in the current
 *     device's context (cudaGetSymbolAddress); the first lookup may load the
 *     library's device code, so make the first call on a device before any
 *     stream capture.
 *   - Every call on a device shares the array and leaves its states there.
 *     Nothing in it needs to start at zero: the second pass reads only states
 *     the first pass of the same call wrote.  Calls whose kernels overlap on
 *     the GPU (different streams, or graphs launched concurrently) race on the
 *     array: serialise them.
 */
#define SOFTMAX_NOALLOC_MAX_STATES 65536
int softmax_fwd_noalloc(const void *in, void *out, int64_t rows, int64_t cols, int64_t row_stride,
                        int dtype, cudaStream_t stream);

/*
 * Shape-keyed autotune.  (Page "GPU Kernels - Implementing and optimizing
 * Softmax", section "Autotuning": try the launch configurations on the real
 * shape and keep the fastest.)
 *
 * softmax_autotune times every candidate launch shape for these arguments
 * (softmax_tune_candidates) on the caller's buffers -- `iters` launches each
 * after two warm-up launches, between CUDA events on `stream` -- and keeps the
 * fastest (another shape displaces the automatic choice only when it is at
 * least 2% faster) in a process-wide cache keyed by (device, dtype, cols, row_stride,
 * in and out address modulo 16, floor(log2(rows))).  From then on softmax_fwd
 * and softmax_plan use the cached shape for every call with that key (a
 * shape forced with softmax_set_force_path still wins).  The automatic choice
 * is always one of the candidates, so the cached shape is never slower than
 * it was in the tuning run.
 *   - in and out must not be the same buffer (the candidates are run many
 *     times and must all see the same input); `out` receives the softmax.
 *   - The call synchronises `stream` and must not be made while the stream is
 *     being captured (SOFTMAX_ERR_ARG).  iters <= 0 means 20.
 *   - The candidates run on the same buffers again and again, so inputs that
 *     fit in L2 are timed warm (as they are when a producer kernel has just
 *     written them).
 *   - result (may be NULL) receives the winning plan, its time and the
 *     automatic plan's time in microseconds per call, and the number of
 *     candidates timed.
 * Returns a softmax_status_t (SOFTMAX_ERR_CUDA if a launch or an event failed;
 * the cache is then unchanged).
 */
typedef struct {
    softmax_plan_t plan;   /* the shape kept */
    double best_us;        /* its time per call */
    double auto_us;        /* the automatic shape's time per call */
    int candidates;        /* shapes timed */
} softmax_tune_result_t;
int softmax_autotune(const void *in, void *out, int64_t rows, int64_t cols, int64_t row_stride,
                     int dtype, cudaStream_t stream, int iters, softmax_tune_result_t *result);

/* One launch shape: path (softmax_path_t) and the threads / vpt / group that
 * softmax_set_force_path takes (0 = the planner's choice). */
typedef struct {
    int path, threads, vpt, group;
} softmax_shape_t;

/*
 * The candidate shapes softmax_autotune would time for these arguments
 * (host only, like softmax_plan with num_sms > 0; num_sms <= 0 asks the
 * current device).  Writes at most `capacity` shapes to `shapes` (the first
 * is always the automatic choice, {0, 0, 0, 0}) and returns how many there
 * are, or a negated softmax_status_t on bad arguments.
 */
int softmax_tune_candidates(uint64_t in_addr, uint64_t out_addr, int64_t rows, int64_t cols,
                            int64_t row_stride, int dtype, int num_sms, softmax_shape_t *shapes,
                            int capacity);

/* Number of shapes in the autotune cache, and a call that empties it. */
int softmax_autotune_size(void);
int softmax_autotune_clear(void);

/* Version of this ABI: major * 10000 + minor * 100 + patch (1.1.0 adds the RING
 * path, 1.2.0 softmax_set_launch_overlap, 1.3.0 the STREAM path and
 * softmax_plan_t.whole_vectors, 1.4.0 the autotune calls and softmax_fwd_masked,
 * 1.5.0 the PACKED path and softmax_fwd_host; 2.0.0 removes the RING path and
 * softmax_plan_t.stages, and softmax_fwd no longer takes the SPLIT path or any
 * scratch; 2.1.0 the GRID path; 2.2.0 softmax_masked_copy). */
int softmax_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MBRS_SOFTMAX_H */
