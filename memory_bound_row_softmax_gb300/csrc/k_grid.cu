// k_grid.cu -- path 8 instantiations: a few very long rows spread over the
// whole grid in two launches (chunk states, then outputs), the states kept in
// the output row itself.
#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

namespace {
template <typename T, int THREADS, int VPT>
cudaError_t go(const LaunchArgs &a, int64_t chunks, int64_t chunk_vecs, int64_t grid) {
    const T *in = static_cast<const T *>(a.in);
    T *out = static_cast<T *>(a.out);
    const cudaError_t e = launch_kernel(k_grid_stats<T, THREADS, VPT>, a, grid, THREADS, 0, 0, in, out, a.rows,
                                        a.cols, a.stride, chunks, chunk_vecs);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_grid_apply<T, THREADS, VPT>, a, grid, THREADS, 0, 0, in, out, a.rows, a.cols, a.stride,
                         chunks, chunk_vecs, a.vec_store);
}

template <typename T>
cudaError_t go_shape(const LaunchArgs &a, int threads, int vpt, int64_t chunks, int64_t chunk_vecs, int64_t grid) {
    if (threads == 256 && vpt == 4) return go<T, 256, 4>(a, chunks, chunk_vecs, grid);
    if (threads == 256 && vpt == 8) return go<T, 256, 8>(a, chunks, chunk_vecs, grid);
    if (threads == 512 && vpt == 4) return go<T, 512, 4>(a, chunks, chunk_vecs, grid);
    if (threads == 1024 && vpt == 4) return go<T, 1024, 4>(a, chunks, chunk_vecs, grid);
    return cudaErrorInvalidValue;
}
}  // namespace

bool grid_shape_ok(int threads, int vpt) {
    return (threads == 256 && (vpt == 4 || vpt == 8)) || (vpt == 4 && (threads == 512 || threads == 1024));
}

cudaError_t launch_grid(const LaunchArgs &a, int threads, int vpt, int64_t chunks, int64_t chunk_vecs,
                        int64_t grid) {
    if (a.in == a.out || chunks < 1 || chunk_vecs < 3) return cudaErrorInvalidValue;
    switch (a.dtype) {
        case 0: return go_shape<float>(a, threads, vpt, chunks, chunk_vecs, grid);
        case 1: return go_shape<__half>(a, threads, vpt, chunks, chunk_vecs, grid);
        case 2: return go_shape<__nv_bfloat16>(a, threads, vpt, chunks, chunk_vecs, grid);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mbrs
