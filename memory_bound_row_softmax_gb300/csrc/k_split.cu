// k_split.cu -- path 4 instantiations: rows split over the grid, two passes.
#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

namespace {
template <typename T, int THREADS, int VPT>
cudaError_t go(const LaunchArgs &a, int64_t chunks, int64_t chunk_vecs, int64_t grid, void *scratch) {
    float2 *part = static_cast<float2 *>(scratch);
    cudaError_t e = launch_kernel(k_split_stats<T, THREADS, VPT>, a, grid, THREADS, 0, 0,
                                  static_cast<const T *>(a.in), a.rows, a.cols, a.stride, chunks, chunk_vecs, part);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_split_apply<T, THREADS, VPT>, a, grid, THREADS, 0, 0,
                         static_cast<const T *>(a.in), static_cast<T *>(a.out), a.rows, a.cols, a.stride, chunks,
                         chunk_vecs, part, a.vec_store);
}

template <typename T>
cudaError_t by_shape(const LaunchArgs &a, int threads, int vpt, int64_t chunks, int64_t chunk_vecs, int64_t grid,
                     void *scratch) {
    if (threads == 256 && vpt == 4) return go<T, 256, 4>(a, chunks, chunk_vecs, grid, scratch);
    if (threads == 512 && vpt == 4) return go<T, 512, 4>(a, chunks, chunk_vecs, grid, scratch);
    if (threads == 256 && vpt == 8) return go<T, 256, 8>(a, chunks, chunk_vecs, grid, scratch);
    return cudaErrorInvalidValue;
}
}  // namespace

bool split_shape_ok(int threads, int vpt) {
    return (threads == 256 && (vpt == 4 || vpt == 8)) || (threads == 512 && vpt == 4);
}

cudaError_t launch_split(const LaunchArgs &a, int threads, int vpt, int64_t chunks, int64_t chunk_vecs,
                         int64_t grid, void *scratch) {
    switch (a.dtype) {
        case 0: return by_shape<float>(a, threads, vpt, chunks, chunk_vecs, grid, scratch);
        case 1: return by_shape<__half>(a, threads, vpt, chunks, chunk_vecs, grid, scratch);
        case 2: return by_shape<__nv_bfloat16>(a, threads, vpt, chunks, chunk_vecs, grid, scratch);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mbrs
