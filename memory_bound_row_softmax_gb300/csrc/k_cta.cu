// k_cta.cu -- path 2 instantiations: a thread block per row.
#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

namespace {
template <typename T, int THREADS, int VPT>
cudaError_t go(const LaunchArgs &a, int64_t grid) {
    if constexpr (VPT >= 6)
        return launch_kernel(k_cta_rows_wide<T, THREADS, VPT>, a, grid, THREADS, 0, 0,
                             static_cast<const T *>(a.in), static_cast<T *>(a.out), a.rows, a.cols, a.stride,
                             a.vec_store);
    else
        return launch_kernel(k_cta_rows<T, THREADS, VPT>, a, grid, THREADS, 0, 0, static_cast<const T *>(a.in),
                             static_cast<T *>(a.out), a.rows, a.cols, a.stride, a.vec_store);
}

template <typename T, int THREADS>
cudaError_t by_vpt(const LaunchArgs &a, int vpt, int64_t grid) {
    switch (vpt) {
        case 1: return go<T, THREADS, 1>(a, grid);
        case 2: return go<T, THREADS, 2>(a, grid);
        case 3: return go<T, THREADS, 3>(a, grid);
        case 4: return go<T, THREADS, 4>(a, grid);
        case 5: return go<T, THREADS, 5>(a, grid);
        default: break;
    }
    if constexpr (THREADS < 1024) {  // 1024 threads x more than 5 vectors would spill
        switch (vpt) {
            case 6: return go<T, THREADS, 6>(a, grid);
            case 8: return go<T, THREADS, 8>(a, grid);
            case 10: return go<T, THREADS, 10>(a, grid);
            default: break;
        }
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t by_shape(const LaunchArgs &a, int threads, int vpt, int64_t grid) {
    switch (threads) {
        case 64: return by_vpt<T, 64>(a, vpt, grid);
        case 128: return by_vpt<T, 128>(a, vpt, grid);
        case 256: return by_vpt<T, 256>(a, vpt, grid);
        case 512: return by_vpt<T, 512>(a, vpt, grid);
        case 1024: return by_vpt<T, 1024>(a, vpt, grid);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

bool cta_shape_ok(int threads, int vpt) {
    const bool t = threads == 64 || threads == 128 || threads == 256 || threads == 512 || threads == 1024;
    return t && ((vpt >= 1 && vpt <= 5) || ((vpt == 6 || vpt == 8 || vpt == 10) && threads < 1024));
}

cudaError_t launch_cta(const LaunchArgs &a, int threads, int vpt, int64_t grid) {
    switch (a.dtype) {
        case 0: return by_shape<float>(a, threads, vpt, grid);
        case 1: return by_shape<__half>(a, threads, vpt, grid);
        case 2: return by_shape<__nv_bfloat16>(a, threads, vpt, grid);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mbrs
