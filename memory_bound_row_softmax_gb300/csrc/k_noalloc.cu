// k_noalloc.cu -- the split (two-pass) path with its per-chunk states in a
// fixed device array instead of memory allocated per call.
//
// Why it exists: softmax_fwd takes the split path's scratch from a stream-
// ordered memory pool.  Some callers cannot allocate device memory at all:
// code running under an allocator that a host framework owns exclusively,
// real-time loops where an allocation's latency or failure is not acceptable,
// or code that must not grow the process's device footprint after start-up.
// softmax_fwd_noalloc serves them: the scratch is the array below, which every
// GPU that loads this library holds from load until process exit.
#include <mutex>

#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

// The scratch of every softmax_fwd_noalloc call on this device: one (s, l)
// state per (row, chunk).  Its size is the hard limit on rows * chunks.
static __device__ __align__(256) float2 g_noalloc_states[kNoAllocMaxStates];

namespace {
constexpr int kMaxDevices = 64;

// Device address of g_noalloc_states on `device` (which must be current).  In
// host code the array's name is only a host-side stand-in, so the address
// comes from cudaGetSymbolAddress, once per device, and is cached.
cudaError_t states_address(int device, float2 **ptr) {
    static std::mutex mu;
    static float2 *addr[kMaxDevices] = {};
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[device]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_states);
        if (e != cudaSuccess) return e;
        addr[device] = static_cast<float2 *>(p);
    }
    *ptr = addr[device];
    return cudaSuccess;
}

template <typename T>
cudaError_t go(const LaunchArgs &a, int64_t chunks, int64_t chunk_vecs, int64_t grid, float2 *states) {
    constexpr int kThreads = kNoAllocThreads, kVpt = kNoAllocVpt;
    cudaError_t e = launch_kernel(k_split_stats<T, kThreads, kVpt>, a, grid, kThreads, 0, 0,
                                  static_cast<const T *>(a.in), a.rows, a.cols, a.stride, chunks, chunk_vecs, states);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_split_apply<T, kThreads, kVpt>, a, grid, kThreads, 0, 0,
                         static_cast<const T *>(a.in), static_cast<T *>(a.out), a.rows, a.cols, a.stride, chunks,
                         chunk_vecs, states, a.vec_store);
}
}  // namespace

cudaError_t launch_split_noalloc(const LaunchArgs &a, int64_t chunks, int64_t chunk_vecs, int64_t grid) {
    if (chunks < 1 || a.rows > kNoAllocMaxStates / chunks) return cudaErrorInvalidValue;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    float2 *states = nullptr;
    if (e == cudaSuccess) e = states_address(device, &states);
    if (e != cudaSuccess) return e;
    switch (a.dtype) {
        case 0: return go<float>(a, chunks, chunk_vecs, grid, states);
        case 1: return go<__half>(a, chunks, chunk_vecs, grid, states);
        case 2: return go<__nv_bfloat16>(a, chunks, chunk_vecs, grid, states);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mbrs
