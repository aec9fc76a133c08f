// warp_launch.cuh -- path 1 launch dispatch, shared by k_warp.cu (rows with
// partial 16-byte vectors), k_warp_whole.cu (rows of whole vectors only),
// k_masked_warp.cu and k_masked_warp_whole.cu (scaled, causally masked rows),
// which instantiate the four variants in separate translation units.
#pragma once

#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

namespace warp_detail {
template <typename T, int G, int VPT, int VAR>
cudaError_t go(const LaunchArgs &a, int threads, int64_t grid) {
    if constexpr (VAR == kMaskedRows || VAR == kMaskedWholeRows)
        return launch_kernel(k_warp_rows_masked<T, G, VPT, VAR == kMaskedWholeRows>, a, grid, threads, 0, 0,
                             static_cast<const T *>(a.in), static_cast<T *>(a.out), a.rows, a.cols, a.stride,
                             a.vec_store, a.mask);
    else
        return launch_kernel(k_warp_rows<T, G, VPT, VAR == kWholeRows>, a, grid, threads, 0, 0,
                             static_cast<const T *>(a.in), static_cast<T *>(a.out), a.rows, a.cols, a.stride,
                             a.vec_store);
}

template <typename T, int G, int VAR>
cudaError_t small_vpt(const LaunchArgs &a, int threads, int vpt, int64_t grid) {
    switch (vpt) {
        case 1: return go<T, G, 1, VAR>(a, threads, grid);
        case 2: return go<T, G, 2, VAR>(a, threads, grid);
        case 3: return go<T, G, 3, VAR>(a, threads, grid);
        case 4: return go<T, G, 4, VAR>(a, threads, grid);
        case 5: return go<T, G, 5, VAR>(a, threads, grid);
        case 6: return go<T, G, 6, VAR>(a, threads, grid);
        case 7: return go<T, G, 7, VAR>(a, threads, grid);
        case 8: return go<T, G, 8, VAR>(a, threads, grid);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, int VAR>
cudaError_t by_shape(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid) {
    switch (group) {
        case 2: return small_vpt<T, 2, VAR>(a, threads, vpt, grid);
        case 4: return small_vpt<T, 4, VAR>(a, threads, vpt, grid);
        case 8: return small_vpt<T, 8, VAR>(a, threads, vpt, grid);
        case 16: return small_vpt<T, 16, VAR>(a, threads, vpt, grid);
        case 32: break;
        default: return cudaErrorInvalidValue;
    }
    switch (vpt) {
        case 1: return go<T, 32, 1, VAR>(a, threads, grid);
        case 2: return go<T, 32, 2, VAR>(a, threads, grid);
        case 3: return go<T, 32, 3, VAR>(a, threads, grid);
        case 4: return go<T, 32, 4, VAR>(a, threads, grid);
        case 5: return go<T, 32, 5, VAR>(a, threads, grid);
        case 6: return go<T, 32, 6, VAR>(a, threads, grid);
        case 7: return go<T, 32, 7, VAR>(a, threads, grid);
        case 8: return go<T, 32, 8, VAR>(a, threads, grid);
        case 9: return go<T, 32, 9, VAR>(a, threads, grid);
        default: return cudaErrorInvalidValue;
    }
}

template <int VAR>
cudaError_t launch(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid) {
    switch (a.dtype) {
        case 0: return by_shape<float, VAR>(a, threads, group, vpt, grid);
        case 1: return by_shape<__half, VAR>(a, threads, group, vpt, grid);
        case 2: return by_shape<__nv_bfloat16, VAR>(a, threads, group, vpt, grid);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace warp_detail

}  // namespace mbrs
