// attention_abi.cu -- the C ABI of the fused attention forward declared in
// include/mbrs_attention.h: argument checks, then the persistent launch
// (k_attention.cu).
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

int softmax_attention_fwd(const void *q, const void *k, const void *v, void *o, int64_t batch, int64_t heads,
                          int64_t n_ctx, int64_t head_dim, int dtype, int causal, float sm_scale,
                          cudaStream_t stream) {
    if (batch < 0 || heads < 0 || n_ctx < 0 || head_dim < 1) return SOFTMAX_ERR_SHAPE;
    if (dtype != SOFTMAX_F32 && dtype != SOFTMAX_F16 && dtype != SOFTMAX_BF16) return SOFTMAX_ERR_DTYPE;
    if (dtype == SOFTMAX_F32 || head_dim != attn::kAttnHeadDim) return SOFTMAX_ERR_UNSUPPORTED;
    if (causal != 0 && causal != 1) return SOFTMAX_ERR_ARG;
    if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return SOFTMAX_ERR_ARG;
    if (batch == 0 || heads == 0 || n_ctx == 0) return SOFTMAX_OK;
    // index ranges of the kernel: n_ctx and the query-tile count fit int32
    constexpr int64_t kInt = 0x7fffffff;
    if (n_ctx > kInt - 128 || batch > kInt / heads) return SOFTMAX_ERR_SHAPE;
    const int64_t bh = batch * heads;
    const int64_t m_tiles = (n_ctx + 127) / 128;
    if (bh > kInt / m_tiles) return SOFTMAX_ERR_SHAPE;
    const int64_t row_bytes = head_dim * 2;
    if (bh > INT64_MAX / n_ctx || bh * n_ctx > INT64_MAX / row_bytes) return SOFTMAX_ERR_SHAPE;
    const uint64_t bytes = (uint64_t)(bh * n_ctx * row_bytes);
    if (!q || !k || !v || !o) return SOFTMAX_ERR_NULL;
    const uint64_t qa = (uint64_t)(uintptr_t)q, ka = (uint64_t)(uintptr_t)k, va = (uint64_t)(uintptr_t)v,
                   oa = (uint64_t)(uintptr_t)o;
    if ((qa | ka | va | oa) & 15u) return SOFTMAX_ERR_ALIGN;
    if (qa > UINT64_MAX - bytes || ka > UINT64_MAX - bytes || va > UINT64_MAX - bytes || oa > UINT64_MAX - bytes)
        return SOFTMAX_ERR_SHAPE;
    const auto overlaps = [bytes](uint64_t a, uint64_t b) { return a < b + bytes && b < a + bytes; };
    if (overlaps(oa, qa) || overlaps(oa, ka) || overlaps(oa, va)) return SOFTMAX_ERR_OVERLAP;
    int sms = 0;
    const int st = mbrs::host_device_sms(&sms);
    if (st != SOFTMAX_OK) return st;
    attn::AttnArgs a{q, k, v, o, batch, heads, n_ctx, dtype, causal, sm_scale, stream, sms};
    const cudaError_t e = attn::launch_attention(a, mbrs::host_wait_ns(), g_attn_starve.load());
    return e == cudaSuccess ? SOFTMAX_OK : SOFTMAX_ERR_CUDA;
}

}  // extern "C"
