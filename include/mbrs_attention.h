/*
 * mbrs_attention.h -- C ABI of the fused attention forward on GB300 (sm_103a).
 *
 * The operation (page "Dissecting Memory Bandwidth & SRAM Tiling in Triton:
 * From GEMM to FlashAttention-3", sections "The Mathematical Remedy: Online
 * Softmax Tiling" and "Writing the Kernel in OpenAI Triton"), for every batch
 * b < batch, head h < heads and query i < n_ctx:
 *
 *     s_ij = sm_scale * sum_c Q[b,h,i,c] K[b,h,j,c]
 *     O[b,h,i,:] = sum_j softmax_j(s_ij) V[b,h,j,:]
 *
 * over the keys j < n_ctx, or with causal != 0 over the keys j <= i only.  The
 * score matrix never leaves the chip: scores are formed tile by tile in tensor
 * memory, their softmax is taken with a running max and normaliser per query,
 * and O is accumulated in tensor memory and divided by the normaliser once.
 *
 * Layout: Q, K, V and O are [batch, heads, n_ctx, head_dim] contiguous
 * (element (b,h,i,c) at ((b * heads + h) * n_ctx + i) * head_dim + c), all of
 * the same dtype: SOFTMAX_F16 or SOFTMAX_BF16.  head_dim must be 128 (the
 * pages' benchmark shape); any n_ctx >= 1.
 *
 * Arithmetic: products of the 16-bit inputs accumulated in fp32 on the tensor
 * cores; exp in fp32; the probabilities P rounded to the input dtype for the
 * second product (as the pages' kernel does); O accumulated in fp32, divided
 * by the fp32 normaliser and rounded once to the dtype (round-to-nearest-even).
 *
 * Ownership: the caller owns all four device buffers and the stream.  Every
 * pointer must be 16-byte aligned.  Q, K and V may overlap one another; O may
 * overlap none of them.  The call is asynchronous on `stream`; nothing is
 * allocated on the device.  The kernel is a persistent grid that hands out
 * its work through a pair of device-side counters.  softmax_attention_fwd
 * takes them from one of 64 slots inside the library, in turn by successive
 * calls: at most 64 of its calls may be in flight at the same time on one
 * device (over all streams), and it cannot be captured into a CUDA graph (a
 * captured launch would keep its slot on every replay while later calls
 * cycle through it): called on a stream that is being captured it returns
 * SOFTMAX_ERR_ARG without launching.  softmax_attention_fwd_counter takes
 * the caller's counters instead, and may be captured.
 *
 * Errors (checked on the host before any launch; nothing is launched unless
 * the result is SOFTMAX_OK):
 *   SOFTMAX_ERR_SHAPE       batch, heads or n_ctx < 0, head_dim < 1, or sizes
 *                           beyond the kernel's index range (2^31 - 1 query
 *                           tiles, n_ctx < 2^31 - 128)
 *   SOFTMAX_ERR_UNSUPPORTED head_dim != 128, or dtype SOFTMAX_F32
 *   SOFTMAX_ERR_DTYPE       dtype not a softmax_dtype_t
 *   SOFTMAX_ERR_NULL        a NULL pointer while there is work to do
 *   SOFTMAX_ERR_ALIGN       a pointer not 16-byte aligned
 *   SOFTMAX_ERR_OVERLAP     O overlaps Q, K or V
 *   SOFTMAX_ERR_ARG         causal not 0 or 1, sm_scale not finite and > 0, or
 *                           (softmax_attention_fwd) the stream is being captured
 *   SOFTMAX_ERR_CUDA        the tensor-map encoder, the capture query or the
 *                           launch failed
 * batch * heads * n_ctx == 0 returns SOFTMAX_OK without a launch.  A bounded
 * wait inside the kernel that runs out sets the device error word that
 * softmax_check_device_error() reports as SOFTMAX_ERR_TIMEOUT.
 */
#ifndef MBRS_ATTENTION_H
#define MBRS_ATTENTION_H

#include "mbrs_softmax.h"

#ifdef __cplusplus
extern "C" {
#endif

int softmax_attention_fwd(const void *q, const void *k, const void *v, void *o, int64_t batch, int64_t heads,
                          int64_t n_ctx, int64_t head_dim, int dtype, int causal, float sm_scale,
                          cudaStream_t stream);

/*
 * softmax_attention_fwd_counter -- the same forward with the persistent
 * grid's two work counters in memory the caller owns, for launches captured
 * into CUDA graphs (and for callers that want more than 64 calls in flight).
 *   work_counter  device pointer to two unsigned ints, 8-byte aligned, that
 *                 overlap none of Q, K, V and O; both zero before the first
 *                 call that uses them.  Every call leaves them zero again when
 *                 its kernel ends, so they need no reset between calls.
 * Calls that share one work_counter must not run at the same time (order them
 * on one stream, or in one graph); calls with different counters may.  Other
 * arguments, layout and status codes as softmax_attention_fwd (also
 * SOFTMAX_ERR_NULL / SOFTMAX_ERR_ALIGN / SOFTMAX_ERR_OVERLAP for the counter);
 * it may be called while the stream is being captured.
 */
int softmax_attention_fwd_counter(const void *q, const void *k, const void *v, void *o, int64_t batch,
                                  int64_t heads, int64_t n_ctx, int64_t head_dim, int dtype, int causal,
                                  float sm_scale, unsigned int *work_counter, cudaStream_t stream);

/* The launch softmax_attention_fwd makes for a shape (host only). */
typedef struct {
    int64_t items;        /* work items: 256-query blocks of one head (batch * heads * ceil(n_ctx / 256)) */
    int64_t grid;         /* persistent blocks launched: min(SMs, items) */
    int head_group;       /* heads per group of the item order (their K and V fit 48 MiB of L2) */
    int threads;          /* threads per block */
    int64_t smem_bytes;   /* dynamic shared memory per block */
    int tmem_columns;     /* tensor-memory columns per block */
    double flops;         /* matmul FLOPs of the call: 4 * batch * heads * n_ctx^2 * head_dim, halved when causal */
} softmax_attention_plan_t;

/*
 * Fill *plan with the launch softmax_attention_fwd would make for these
 * arguments on a device with num_sms SMs (num_sms <= 0: the current device's
 * count, which needs the CUDA runtime).  Returns the status the call would
 * return for the shape, dtype, causal and head_dim arguments (pointers are not
 * checked); SOFTMAX_ERR_ARG when plan is NULL.
 */
int softmax_attention_plan(int64_t batch, int64_t heads, int64_t n_ctx, int64_t head_dim, int dtype, int causal,
                           int num_sms, softmax_attention_plan_t *plan);

/*
 * Test hook for the attention forward's bounded waits.  starve != 0 makes the
 * next launches leave every block's first Q barrier unarmed, so that wait can
 * only run out: the kernel records SOFTMAX_ERR_TIMEOUT (read it with
 * softmax_check_device_error), skips its stores and returns normally.  The
 * wait limit is the one softmax_set_wait_test sets (default 1 s).
 * Process-wide, not thread-safe; returns SOFTMAX_OK.
 */
int softmax_attention_set_wait_test(int starve);

#ifdef __cplusplus
}
#endif

#endif /* MBRS_ATTENTION_H */
