// k_pattern_copy.cu -- softmax_masked_copy: the memory traffic of a
// softmax_fwd_masked call with no arithmetic (each row's kept entries read and
// written, the rest of the row zero-filled), a reference time for the masked
// call in the way a same-bytes device-to-device copy is one for softmax_fwd.
#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

namespace {
// Keep the first `bytes` bytes of a 16-byte word (little-endian lanes), zero the rest.
__device__ __forceinline__ uint4 keep_bytes(uint4 w, int bytes) {
    uint32_t *p = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int b = bytes - 4 * i;
        p[i] = b >= 4 ? p[i] : b <= 0 ? 0u : p[i] & ((1u << (8 * b)) - 1u);
    }
    return w;
}

// One block per row (grid-stride over rows); rows of whole 16-byte vectors.
// A thread loads up to VPT kept vectors of a span, then stores the span.
template <int VPT>
__global__ void __launch_bounds__(1024) k_masked_copy(const uint4 *__restrict__ in, uint4 *__restrict__ out,
                                                      int64_t rows, int64_t cols, int64_t svec, int es,
                                                      CausalMask mask) {
    pdl_enter();
    const int V = kVecBytes / es;
    const int64_t nvec = cols / V, span = (int64_t)blockDim.x * VPT;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t kept = mask.kept(row, cols), kv = kept / V;
        const int rem_bytes = (int)(kept % V) * es;  // kept bytes of vector kv
        const uint4 *src = in + row * svec;
        uint4 *dst = out + row * svec;
        for (int64_t base = 0; base < nvec; base += span) {
            uint4 r[VPT];
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int64_t v = base + threadIdx.x + (int64_t)j * blockDim.x;
                r[j] = make_uint4(0u, 0u, 0u, 0u);
                if (v < kv || (v == kv && rem_bytes > 0)) r[j] = src[v];
            }
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int64_t v = base + threadIdx.x + (int64_t)j * blockDim.x;
                if (v < nvec) dst[v] = v == kv ? keep_bytes(r[j], rem_bytes) : r[j];
            }
        }
    }
}
}  // namespace

cudaError_t launch_masked_copy(const LaunchArgs &a, int threads, int64_t grid) {
    const int es = a.dtype == 0 ? 4 : 2;
    const int64_t svec = a.stride * es / kVecBytes;
    return launch_kernel(k_masked_copy<8>, a, grid, threads, 0, 0, static_cast<const uint4 *>(a.in),
                         static_cast<uint4 *>(a.out), a.rows, a.cols, svec, es, a.mask);
}

}  // namespace mbrs
