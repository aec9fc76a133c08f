// attention_abi.cu -- the C ABI of the fused attention forward declared in
// include/mbrs_attention.h: argument checks, then the persistent launch
// (k_attention.cu).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "mbrs_attention.h"
#include "attention_launch.h"
#include "launch.h"

using namespace mbrs;

namespace {
std::atomic<int> g_attn_starve{0};
}

extern "C" {

int softmax_attention_set_wait_test(int starve) {
    g_attn_starve.store(starve ? 1 : 0);
    return SOFTMAX_OK;
}

namespace {

// The checks of everything but the pointers, shared by the call and its plan.
int check_shape(int64_t batch, int64_t heads, int64_t n_ctx, int64_t head_dim, int dtype, int causal) {
    if (batch < 0 || heads < 0 || n_ctx < 0 || head_dim < 1) return SOFTMAX_ERR_SHAPE;
    if (dtype != SOFTMAX_F32 && dtype != SOFTMAX_F16 && dtype != SOFTMAX_BF16) return SOFTMAX_ERR_DTYPE;
    if (dtype == SOFTMAX_F32 || head_dim != attn::kAttnHeadDim) return SOFTMAX_ERR_UNSUPPORTED;
    if (causal != 0 && causal != 1) return SOFTMAX_ERR_ARG;
    if (batch == 0 || heads == 0 || n_ctx == 0) return SOFTMAX_OK;
    // index ranges of the kernel: n_ctx and the query-tile count fit int32
    constexpr int64_t kInt = 0x7fffffff;
    if (n_ctx > kInt - 128 || batch > kInt / heads) return SOFTMAX_ERR_SHAPE;
    const int64_t bh = batch * heads;
    const int64_t m_tiles = (n_ctx + 127) / 128;
    if (bh > kInt / m_tiles) return SOFTMAX_ERR_SHAPE;
    const int64_t row_bytes = head_dim * 2;
    if (bh > INT64_MAX / n_ctx || bh * n_ctx > INT64_MAX / row_bytes) return SOFTMAX_ERR_SHAPE;
    return SOFTMAX_OK;
}

}  // namespace

int softmax_attention_plan(int64_t batch, int64_t heads, int64_t n_ctx, int64_t head_dim, int dtype, int causal,
                           int num_sms, softmax_attention_plan_t *plan) {
    if (!plan) return SOFTMAX_ERR_ARG;
    *plan = softmax_attention_plan_t{};
    const int st = check_shape(batch, heads, n_ctx, head_dim, dtype, causal);
    if (st != SOFTMAX_OK) return st;
    plan->threads = attn::attention_threads();
    plan->smem_bytes = (int64_t)attn::attention_smem_bytes();
    plan->tmem_columns = attn::attention_tmem_columns();
    if (batch == 0 || heads == 0 || n_ctx == 0) return SOFTMAX_OK;
    int sms = num_sms;
    if (sms <= 0) {
        const int e = mbrs::host_device_sms(&sms);
        if (e != SOFTMAX_OK) return e;
    }
    plan->items = attn::attention_items(batch, heads, n_ctx);
    plan->grid = std::min<int64_t>(sms, plan->items);
    plan->head_group = attn::attention_head_group(batch * heads, n_ctx);
    const double f = 4.0 * (double)batch * (double)heads * (double)n_ctx * (double)n_ctx * (double)head_dim;
    plan->flops = causal ? f / 2 : f;
    return SOFTMAX_OK;
}

namespace {

int attention_call(const void *q, const void *k, const void *v, void *o, int64_t batch, int64_t heads,
                   int64_t n_ctx, int64_t head_dim, int dtype, int causal, float sm_scale, unsigned int *counter,
                   cudaStream_t stream) {
    int st = check_shape(batch, heads, n_ctx, head_dim, dtype, causal);
    if (st != SOFTMAX_OK) return st;
    if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return SOFTMAX_ERR_ARG;
    if (batch == 0 || heads == 0 || n_ctx == 0) return SOFTMAX_OK;
    const int64_t bh = batch * heads;
    const uint64_t bytes = (uint64_t)(bh * n_ctx * head_dim * 2);
    if (!q || !k || !v || !o) return SOFTMAX_ERR_NULL;
    const uint64_t qa = (uint64_t)(uintptr_t)q, ka = (uint64_t)(uintptr_t)k, va = (uint64_t)(uintptr_t)v,
                   oa = (uint64_t)(uintptr_t)o;
    if ((qa | ka | va | oa) & 15u) return SOFTMAX_ERR_ALIGN;
    if (qa > UINT64_MAX - bytes || ka > UINT64_MAX - bytes || va > UINT64_MAX - bytes || oa > UINT64_MAX - bytes)
        return SOFTMAX_ERR_SHAPE;
    const auto overlaps = [bytes](uint64_t a, uint64_t b) { return a < b + bytes && b < a + bytes; };
    if (overlaps(oa, qa) || overlaps(oa, ka) || overlaps(oa, va)) return SOFTMAX_ERR_OVERLAP;
    if (counter) {  // the counter's 8 bytes are written: they may overlap no tensor
        const uint64_t ca = (uint64_t)(uintptr_t)counter;
        const auto hits = [bytes, ca](uint64_t a) { return ca < a + bytes && a < ca + 8; };
        if (hits(qa) || hits(ka) || hits(va) || hits(oa)) return SOFTMAX_ERR_OVERLAP;
    } else {
        // a captured launch would keep the library slot it took at capture on
        // every replay, sharing it with whatever later call takes that slot:
        // captures must bring their own counter (softmax_attention_fwd_counter)
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return SOFTMAX_ERR_CUDA;
        if (cap != cudaStreamCaptureStatusNone) return SOFTMAX_ERR_ARG;
    }
    int sms = 0;
    st = mbrs::host_device_sms(&sms);
    if (st != SOFTMAX_OK) return st;
    attn::AttnArgs a{q, k, v, o, batch, heads, n_ctx, dtype, causal, sm_scale, stream, sms, counter};
    const cudaError_t e = attn::launch_attention(a, mbrs::host_wait_ns(), g_attn_starve.load());
    return e == cudaSuccess ? SOFTMAX_OK : SOFTMAX_ERR_CUDA;
}

}  // namespace

int softmax_attention_fwd(const void *q, const void *k, const void *v, void *o, int64_t batch, int64_t heads,
                          int64_t n_ctx, int64_t head_dim, int dtype, int causal, float sm_scale,
                          cudaStream_t stream) {
    return attention_call(q, k, v, o, batch, heads, n_ctx, head_dim, dtype, causal, sm_scale, nullptr, stream);
}

int softmax_attention_fwd_counter(const void *q, const void *k, const void *v, void *o, int64_t batch,
                                  int64_t heads, int64_t n_ctx, int64_t head_dim, int dtype, int causal,
                                  float sm_scale, unsigned int *work_counter, cudaStream_t stream) {
    const int st = check_shape(batch, heads, n_ctx, head_dim, dtype, causal);
    if (st != SOFTMAX_OK) return st;
    if (batch == 0 || heads == 0 || n_ctx == 0) return SOFTMAX_OK;
    if (!work_counter) return SOFTMAX_ERR_NULL;
    if ((uintptr_t)work_counter % 8 != 0) return SOFTMAX_ERR_ALIGN;
    return attention_call(q, k, v, o, batch, heads, n_ctx, head_dim, dtype, causal, sm_scale, work_counter,
                          stream);
}

}  // extern "C"
