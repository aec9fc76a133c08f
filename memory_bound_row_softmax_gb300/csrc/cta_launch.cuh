// cta_launch.cuh -- path 2 launch dispatch, shared by k_cta.cu (rows with
// partial 16-byte vectors), k_cta_whole.cu (rows of whole vectors only),
// k_masked.cu and k_masked_whole.cu (scaled, causally masked rows), which
// instantiate the four variants in separate translation units.
#pragma once

#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

namespace cta_detail {
template <typename T, int THREADS, int VPT, int VAR>
cudaError_t go(const LaunchArgs &a, int64_t grid) {
    constexpr bool whole = VAR == kWholeRows || VAR == kMaskedWholeRows;
    constexpr bool masked = VAR == kMaskedRows || VAR == kMaskedWholeRows;
    if constexpr (masked && VPT >= 6)
        return launch_kernel(k_cta_rows_masked_wide<T, THREADS, VPT, whole>, a, grid, THREADS, 0, 0,
                             static_cast<const T *>(a.in), static_cast<T *>(a.out), a.rows, a.cols, a.stride,
                             a.vec_store, a.mask);
    else if constexpr (masked)
        return launch_kernel(k_cta_rows_masked<T, THREADS, VPT, whole>, a, grid, THREADS, 0, 0,
                             static_cast<const T *>(a.in), static_cast<T *>(a.out), a.rows, a.cols, a.stride,
                             a.vec_store, a.mask);
    else if constexpr (VPT >= 6)
        return launch_kernel(k_cta_rows_wide<T, THREADS, VPT, whole>, a, grid, THREADS, 0, 0,
                             static_cast<const T *>(a.in), static_cast<T *>(a.out), a.rows, a.cols, a.stride,
                             a.vec_store);
    else
        return launch_kernel(k_cta_rows<T, THREADS, VPT, whole>, a, grid, THREADS, 0, 0, static_cast<const T *>(a.in),
                             static_cast<T *>(a.out), a.rows, a.cols, a.stride, a.vec_store);
}

template <typename T, int THREADS, int VAR>
cudaError_t by_vpt(const LaunchArgs &a, int vpt, int64_t grid) {
    switch (vpt) {
        case 1: return go<T, THREADS, 1, VAR>(a, grid);
        case 2: return go<T, THREADS, 2, VAR>(a, grid);
        case 3: return go<T, THREADS, 3, VAR>(a, grid);
        case 4: return go<T, THREADS, 4, VAR>(a, grid);
        case 5: return go<T, THREADS, 5, VAR>(a, grid);
        default: break;
    }
    if constexpr (THREADS < 1024) {  // 1024 threads x more than 5 vectors would spill
        switch (vpt) {
            case 6: return go<T, THREADS, 6, VAR>(a, grid);
            case 8: return go<T, THREADS, 8, VAR>(a, grid);
            case 10: return go<T, THREADS, 10, VAR>(a, grid);
            default: break;
        }
    }
    return cudaErrorInvalidValue;
}

template <typename T, int VAR>
cudaError_t by_shape(const LaunchArgs &a, int threads, int vpt, int64_t grid) {
    switch (threads) {
        case 64: return by_vpt<T, 64, VAR>(a, vpt, grid);
        case 128: return by_vpt<T, 128, VAR>(a, vpt, grid);
        case 256: return by_vpt<T, 256, VAR>(a, vpt, grid);
        case 512: return by_vpt<T, 512, VAR>(a, vpt, grid);
        case 1024: return by_vpt<T, 1024, VAR>(a, vpt, grid);
        default: return cudaErrorInvalidValue;
    }
}

template <int VAR>
cudaError_t launch(const LaunchArgs &a, int threads, int vpt, int64_t grid) {
    switch (a.dtype) {
        case 0: return by_shape<float, VAR>(a, threads, vpt, grid);
        case 1: return by_shape<__half, VAR>(a, threads, vpt, grid);
        case 2: return by_shape<__nv_bfloat16, VAR>(a, threads, vpt, grid);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace cta_detail

}  // namespace mbrs
