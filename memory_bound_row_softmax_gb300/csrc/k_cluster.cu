// k_cluster.cu -- path 3 instantiations: a thread-block cluster per row, each
// block holding its slice in registers, with a (max, sum) exchange through
// distributed shared memory; path 6, the same cluster streaming slices of any
// length in two passes.  Also reads and clears the device error word.
#include <atomic>

#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

namespace {
constexpr int kMaxDevices = 64;

// per kernel and device, once: opt in to `smem` bytes of dynamic shared
// memory and to clusters of up to 16 blocks
template <typename K>
cudaError_t opt_in(K fn, int smem, std::atomic<unsigned long long> &done, int device) {
    const unsigned long long bit = 1ull << (device & (kMaxDevices - 1));
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

template <typename T, int THREADS, int VPT, bool WHOLE>
cudaError_t go_as(const LaunchArgs &a, int csize, int64_t wait_ns, int starve) {
    static std::atomic<unsigned long long> done{0};
    constexpr int smem = ClusterSmem<THREADS>::kBytes;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e == cudaSuccess) e = opt_in(k_cluster_rows<T, THREADS, VPT, WHOLE>, smem, done, device);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_cluster_rows<T, THREADS, VPT, WHOLE>, a, a.rows * csize, THREADS, smem, csize,
                         static_cast<const T *>(a.in), static_cast<T *>(a.out), a.rows, a.cols, a.stride,
                         a.vec_store, wait_ns, starve);
}

// 16-bit rows, 8 vectors per thread held in registers (fp32 at 8 vectors
// would spill at the 64 registers two 512-thread blocks per SM allow)
template <typename T>
cudaError_t by_shape(const LaunchArgs &a, int threads, int vpt, int csize, int64_t wait_ns, int starve) {
    if constexpr (sizeof(T) == 2) {
        if (vpt != 8) return cudaErrorInvalidValue;
        switch (threads) {
            case 256: return a.whole ? go_as<T, 256, 8, true>(a, csize, wait_ns, starve)
                                     : go_as<T, 256, 8, false>(a, csize, wait_ns, starve);
            case 512: return a.whole ? go_as<T, 512, 8, true>(a, csize, wait_ns, starve)
                                     : go_as<T, 512, 8, false>(a, csize, wait_ns, starve);
            default: return cudaErrorInvalidValue;
        }
    }
    return cudaErrorInvalidValue;
}

// path 6: the streaming two-pass cluster kernel
template <typename T, int THREADS, int VPT, bool WHOLE>
cudaError_t stream_as(const LaunchArgs &a, int csize, int64_t wait_ns, int starve) {
    static std::atomic<unsigned long long> done{0};
    constexpr int smem = ClusterSmem<THREADS>::kBytes;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e == cudaSuccess) e = opt_in(k_cluster_stream<T, THREADS, VPT, WHOLE>, smem, done, device);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_cluster_stream<T, THREADS, VPT, WHOLE>, a, a.rows * csize, THREADS, smem, csize,
                         static_cast<const T *>(a.in), static_cast<T *>(a.out), a.rows, a.cols, a.stride,
                         a.vec_store, wait_ns, starve);
}

// masked rows (softmax_fwd_masked)
template <typename T, int THREADS, int VPT, bool WHOLE>
cudaError_t stream_masked_as(const LaunchArgs &a, int csize, int64_t wait_ns, int starve) {
    static std::atomic<unsigned long long> done{0};
    constexpr int smem = ClusterSmem<THREADS>::kBytes;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e == cudaSuccess) e = opt_in(k_cluster_stream_masked<T, THREADS, VPT, WHOLE>, smem, done, device);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_cluster_stream_masked<T, THREADS, VPT, WHOLE>, a, a.rows * csize, THREADS, smem, csize,
                         static_cast<const T *>(a.in), static_cast<T *>(a.out), a.rows, a.cols, a.stride,
                         a.vec_store, wait_ns, starve, a.mask);
}

template <typename T, int THREADS, bool MASKED>
cudaError_t stream_vpt(const LaunchArgs &a, int vpt, int csize, int64_t wait_ns, int starve) {
    if constexpr (MASKED) {
        switch (vpt) {
            case 2: return a.whole ? stream_masked_as<T, THREADS, 2, true>(a, csize, wait_ns, starve)
                                   : stream_masked_as<T, THREADS, 2, false>(a, csize, wait_ns, starve);
            case 4: return a.whole ? stream_masked_as<T, THREADS, 4, true>(a, csize, wait_ns, starve)
                                   : stream_masked_as<T, THREADS, 4, false>(a, csize, wait_ns, starve);
            default: return cudaErrorInvalidValue;
        }
    } else {
        switch (vpt) {
            case 2: return a.whole ? stream_as<T, THREADS, 2, true>(a, csize, wait_ns, starve)
                                   : stream_as<T, THREADS, 2, false>(a, csize, wait_ns, starve);
            case 4: return a.whole ? stream_as<T, THREADS, 4, true>(a, csize, wait_ns, starve)
                                   : stream_as<T, THREADS, 4, false>(a, csize, wait_ns, starve);
            default: return cudaErrorInvalidValue;
        }
    }
}

template <typename T, bool MASKED>
cudaError_t stream_shape(const LaunchArgs &a, int threads, int vpt, int csize, int64_t wait_ns, int starve) {
    switch (threads) {
        case 256: return stream_vpt<T, 256, MASKED>(a, vpt, csize, wait_ns, starve);
        case 512: return stream_vpt<T, 512, MASKED>(a, vpt, csize, wait_ns, starve);
        case 1024: return stream_vpt<T, 1024, MASKED>(a, vpt, csize, wait_ns, starve);
        default: return cudaErrorInvalidValue;
    }
}

template <bool MASKED>
cudaError_t stream_dtype(const LaunchArgs &a, int threads, int vpt, int csize, int64_t wait_ns, int starve) {
    if (csize < 1 || csize > kMaxCluster) return cudaErrorInvalidValue;
    switch (a.dtype) {
        case 0: return stream_shape<float, MASKED>(a, threads, vpt, csize, wait_ns, starve);
        case 1: return stream_shape<__half, MASKED>(a, threads, vpt, csize, wait_ns, starve);
        case 2: return stream_shape<__nv_bfloat16, MASKED>(a, threads, vpt, csize, wait_ns, starve);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

bool stream_shape_ok(int threads, int vpt) {
    return (threads == 256 || threads == 512 || threads == 1024) && (vpt == 2 || vpt == 4);
}

int64_t stream_smem_bytes(int threads) { return 16 + (threads / 32) * 8 + kMaxCluster * 8; }

cudaError_t launch_stream(const LaunchArgs &a, int threads, int vpt, int csize, int64_t wait_ns, int starve) {
    return stream_dtype<false>(a, threads, vpt, csize, wait_ns, starve);
}

cudaError_t launch_stream_masked(const LaunchArgs &a, int threads, int vpt, int csize, int64_t wait_ns,
                                 int starve) {
    return stream_dtype<true>(a, threads, vpt, csize, wait_ns, starve);
}

bool cluster_shape_ok(int threads, int vpt, int elem_bytes) {
    return (threads == 256 || threads == 512) && vpt == 8 && elem_bytes == 2;
}

int64_t cluster_smem_bytes(int threads) { return 16 + (threads / 32) * 8 + kMaxCluster * 8; }

cudaError_t launch_cluster(const LaunchArgs &a, int threads, int vpt, int csize, int64_t wait_ns, int starve) {
    if (csize < 1 || csize > kMaxCluster) return cudaErrorInvalidValue;
    switch (a.dtype) {
        case 0: return by_shape<float>(a, threads, vpt, csize, wait_ns, starve);
        case 1: return by_shape<__half>(a, threads, vpt, csize, wait_ns, starve);
        case 2: return by_shape<__nv_bfloat16>(a, threads, vpt, csize, wait_ns, starve);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_clear_error_word(cudaStream_t stream, unsigned int *word) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(word, g_error_word, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(unsigned int), 0, cudaMemcpyHostToDevice);
}

}  // namespace mbrs
