// attention_launch.h -- host-side interface of the fused attention forward
// (k_attention.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mbrs {
namespace attn {

constexpr int kAttnHeadDim = 128;  // the one head dimension the kernel is built for
constexpr int kAttnF16 = 1, kAttnBf16 = 2;

// Q, K, V, O: [batch, heads, n_ctx, kAttnHeadDim] contiguous, 16-byte
// aligned, of dtype kAttnF16 or kAttnBf16.  The caller has checked them.
struct AttnArgs {
    const void *q, *k, *v;
    void *o;
    int64_t batch, heads, n_ctx;
    int dtype;
    int causal;
    float sm_scale;
    cudaStream_t stream;
    int sms;  // the device's SM count: the persistent grid's size
    unsigned int *counter;  // the caller's two work-counter words, or nullptr: a library slot
};

// starve != 0 (a test hook): every block leaves its first item's Q barrier
// unarmed, so that wait runs out and the whole launch takes its abort path
cudaError_t launch_attention(const AttnArgs &a, int64_t wait_ns, int starve);
// heads per block-order group: as many as keep the group's K and V within
// kAttnGroupBytes (a share of the 126 MB L2), at least 1, at most all
constexpr int64_t kAttnGroupBytes = 48ll << 20;
int attention_head_group(int64_t heads_total, int64_t n_ctx);
// 256-query work items of a call (the persistent grid walks them)
int64_t attention_items(int64_t batch, int64_t heads, int64_t n_ctx);
size_t attention_smem_bytes();
int attention_threads();
int attention_tmem_columns();
// the attention kernel's device error word (kErrWaitTimeout when a bounded
// wait ran out); read after the stream has been synchronised, then cleared
cudaError_t read_clear_attn_error_word(unsigned int *word);

}  // namespace attn
}  // namespace mbrs
