// warp_launch.cuh -- path 1 launch dispatch, shared by k_warp.cu (rows with
// partial 16-byte vectors) and k_warp_whole.cu (rows of whole vectors only),
// which instantiate the two halves in separate translation units.
#pragma once

#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

namespace warp_detail {
template <typename T, int G, int VPT, bool WHOLE>
cudaError_t go(const LaunchArgs &a, int threads, int64_t grid) {
    return launch_kernel(k_warp_rows<T, G, VPT, WHOLE>, a, grid, threads, 0, 0, static_cast<const T *>(a.in),
                         static_cast<T *>(a.out), a.rows, a.cols, a.stride, a.vec_store);
}

template <typename T, int G, bool WHOLE>
cudaError_t small_vpt(const LaunchArgs &a, int threads, int vpt, int64_t grid) {
    switch (vpt) {
        case 1: return go<T, G, 1, WHOLE>(a, threads, grid);
        case 2: return go<T, G, 2, WHOLE>(a, threads, grid);
        case 3: return go<T, G, 3, WHOLE>(a, threads, grid);
        case 4: return go<T, G, 4, WHOLE>(a, threads, grid);
        case 5: return go<T, G, 5, WHOLE>(a, threads, grid);
        case 6: return go<T, G, 6, WHOLE>(a, threads, grid);
        case 7: return go<T, G, 7, WHOLE>(a, threads, grid);
        case 8: return go<T, G, 8, WHOLE>(a, threads, grid);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, bool WHOLE>
cudaError_t by_shape(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid) {
    switch (group) {
        case 2: return small_vpt<T, 2, WHOLE>(a, threads, vpt, grid);
        case 4: return small_vpt<T, 4, WHOLE>(a, threads, vpt, grid);
        case 8: return small_vpt<T, 8, WHOLE>(a, threads, vpt, grid);
        case 16: return small_vpt<T, 16, WHOLE>(a, threads, vpt, grid);
        case 32: break;
        default: return cudaErrorInvalidValue;
    }
    switch (vpt) {
        case 1: return go<T, 32, 1, WHOLE>(a, threads, grid);
        case 2: return go<T, 32, 2, WHOLE>(a, threads, grid);
        case 3: return go<T, 32, 3, WHOLE>(a, threads, grid);
        case 4: return go<T, 32, 4, WHOLE>(a, threads, grid);
        case 5: return go<T, 32, 5, WHOLE>(a, threads, grid);
        case 6: return go<T, 32, 6, WHOLE>(a, threads, grid);
        case 7: return go<T, 32, 7, WHOLE>(a, threads, grid);
        case 8: return go<T, 32, 8, WHOLE>(a, threads, grid);
        case 9: return go<T, 32, 9, WHOLE>(a, threads, grid);
        default: return cudaErrorInvalidValue;
    }
}

template <bool WHOLE>
cudaError_t launch(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid) {
    switch (a.dtype) {
        case 0: return by_shape<float, WHOLE>(a, threads, group, vpt, grid);
        case 1: return by_shape<__half, WHOLE>(a, threads, group, vpt, grid);
        case 2: return by_shape<__nv_bfloat16, WHOLE>(a, threads, group, vpt, grid);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace warp_detail

}  // namespace mbrs
