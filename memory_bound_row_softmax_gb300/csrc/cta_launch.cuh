// cta_launch.cuh -- path 2 launch dispatch, shared by k_cta.cu (rows with
// partial 16-byte vectors) and k_cta_whole.cu (rows of whole vectors only),
// which instantiate the two halves in separate translation units.
#pragma once

#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

namespace cta_detail {
template <typename T, int THREADS, int VPT, bool WHOLE>
cudaError_t go(const LaunchArgs &a, int64_t grid) {
    if constexpr (VPT >= 6)
        return launch_kernel(k_cta_rows_wide<T, THREADS, VPT, WHOLE>, a, grid, THREADS, 0, 0,
                             static_cast<const T *>(a.in), static_cast<T *>(a.out), a.rows, a.cols, a.stride,
                             a.vec_store);
    else
        return launch_kernel(k_cta_rows<T, THREADS, VPT, WHOLE>, a, grid, THREADS, 0, 0, static_cast<const T *>(a.in),
                             static_cast<T *>(a.out), a.rows, a.cols, a.stride, a.vec_store);
}

template <typename T, int THREADS, bool WHOLE>
cudaError_t by_vpt(const LaunchArgs &a, int vpt, int64_t grid) {
    switch (vpt) {
        case 1: return go<T, THREADS, 1, WHOLE>(a, grid);
        case 2: return go<T, THREADS, 2, WHOLE>(a, grid);
        case 3: return go<T, THREADS, 3, WHOLE>(a, grid);
        case 4: return go<T, THREADS, 4, WHOLE>(a, grid);
        case 5: return go<T, THREADS, 5, WHOLE>(a, grid);
        default: break;
    }
    if constexpr (THREADS < 1024) {  // 1024 threads x more than 5 vectors would spill
        switch (vpt) {
            case 6: return go<T, THREADS, 6, WHOLE>(a, grid);
            case 8: return go<T, THREADS, 8, WHOLE>(a, grid);
            case 10: return go<T, THREADS, 10, WHOLE>(a, grid);
            default: break;
        }
    }
    return cudaErrorInvalidValue;
}

template <typename T, bool WHOLE>
cudaError_t by_shape(const LaunchArgs &a, int threads, int vpt, int64_t grid) {
    switch (threads) {
        case 64: return by_vpt<T, 64, WHOLE>(a, vpt, grid);
        case 128: return by_vpt<T, 128, WHOLE>(a, vpt, grid);
        case 256: return by_vpt<T, 256, WHOLE>(a, vpt, grid);
        case 512: return by_vpt<T, 512, WHOLE>(a, vpt, grid);
        case 1024: return by_vpt<T, 1024, WHOLE>(a, vpt, grid);
        default: return cudaErrorInvalidValue;
    }
}

template <bool WHOLE>
cudaError_t launch(const LaunchArgs &a, int threads, int vpt, int64_t grid) {
    switch (a.dtype) {
        case 0: return by_shape<float, WHOLE>(a, threads, vpt, grid);
        case 1: return by_shape<__half, WHOLE>(a, threads, vpt, grid);
        case 2: return by_shape<__nv_bfloat16, WHOLE>(a, threads, vpt, grid);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace cta_detail

}  // namespace mbrs
