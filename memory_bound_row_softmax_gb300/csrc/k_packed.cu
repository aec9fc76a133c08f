// k_packed.cu -- path 7 instantiations: narrow dense rows staged through
// shared memory as contiguous spans, one thread per row.
#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

namespace {
template <typename T>
cudaError_t go(const LaunchArgs &a, int rows_per_span, int64_t grid, int64_t smem) {
    return launch_kernel(k_packed_rows<T>, a, grid, kPackedThreads, (size_t)smem, 0, static_cast<const T *>(a.in),
                         static_cast<T *>(a.out), a.rows, a.cols, rows_per_span);
}
}  // namespace

int64_t packed_smem_bytes(int64_t rows_per_span, int64_t cols, int elem_bytes) {
    const int64_t v = kVecBytes / elem_bytes;
    return (rows_per_span * cols + 2 * v) * 4;
}

cudaError_t launch_packed(const LaunchArgs &a, int rows_per_span, int64_t grid) {
    // dense rows only, out in the same 16-byte phase as in
    if (a.stride != a.cols || !a.vec_store || rows_per_span < 1) return cudaErrorInvalidValue;
    const int64_t smem = packed_smem_bytes(rows_per_span, a.cols, a.dtype == 0 ? 4 : 2);
    if (smem > kPackedMaxSmem) return cudaErrorInvalidValue;
    switch (a.dtype) {
        case 0: return go<float>(a, rows_per_span, grid, smem);
        case 1: return go<__half>(a, rows_per_span, grid, smem);
        case 2: return go<__nv_bfloat16>(a, rows_per_span, grid, smem);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mbrs
