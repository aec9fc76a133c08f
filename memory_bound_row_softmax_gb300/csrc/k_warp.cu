// k_warp.cu -- path 1 instantiations: a lane group (2..32 lanes) per row.
#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

namespace {
template <typename T, int G, int VPT>
cudaError_t go(const LaunchArgs &a, int threads, int64_t grid) {
    return launch_kernel(k_warp_rows<T, G, VPT>, a, grid, threads, 0, 0, static_cast<const T *>(a.in),
                         static_cast<T *>(a.out), a.rows, a.cols, a.stride, a.vec_store);
}

template <typename T, int G>
cudaError_t small_vpt(const LaunchArgs &a, int threads, int vpt, int64_t grid) {
    switch (vpt) {
        case 1: return go<T, G, 1>(a, threads, grid);
        case 2: return go<T, G, 2>(a, threads, grid);
        case 3: return go<T, G, 3>(a, threads, grid);
        case 4: return go<T, G, 4>(a, threads, grid);
        case 5: return go<T, G, 5>(a, threads, grid);
        case 6: return go<T, G, 6>(a, threads, grid);
        case 7: return go<T, G, 7>(a, threads, grid);
        case 8: return go<T, G, 8>(a, threads, grid);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t by_shape(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid) {
    switch (group) {
        case 2: return small_vpt<T, 2>(a, threads, vpt, grid);
        case 4: return small_vpt<T, 4>(a, threads, vpt, grid);
        case 8: return small_vpt<T, 8>(a, threads, vpt, grid);
        case 16: return small_vpt<T, 16>(a, threads, vpt, grid);
        case 32: break;
        default: return cudaErrorInvalidValue;
    }
    switch (vpt) {
        case 1: return go<T, 32, 1>(a, threads, grid);
        case 2: return go<T, 32, 2>(a, threads, grid);
        case 3: return go<T, 32, 3>(a, threads, grid);
        case 4: return go<T, 32, 4>(a, threads, grid);
        case 5: return go<T, 32, 5>(a, threads, grid);
        case 6: return go<T, 32, 6>(a, threads, grid);
        case 7: return go<T, 32, 7>(a, threads, grid);
        case 8: return go<T, 32, 8>(a, threads, grid);
        case 9: return go<T, 32, 9>(a, threads, grid);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

bool warp_shape_ok(int group, int vpt) {
    if (group == 2 || group == 4 || group == 8 || group == 16) return vpt >= 1 && vpt <= 8;
    return group == 32 && vpt >= 1 && vpt <= 9;
}

cudaError_t launch_warp(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid) {
    if (threads < 32 || threads > 256 || threads % 32 != 0) return cudaErrorInvalidValue;
    switch (a.dtype) {
        case 0: return by_shape<float>(a, threads, group, vpt, grid);
        case 1: return by_shape<__half>(a, threads, group, vpt, grid);
        case 2: return by_shape<__nv_bfloat16>(a, threads, group, vpt, grid);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mbrs
