// k_noalloc.cu -- the split (two-pass) path with its per-chunk states in a
// fixed device array instead of memory allocated per call.
//
// Why it exists: the split spreads a few very long rows over the whole GPU,
// and its two passes meet in per-chunk states.  softmax_fwd keeps such states
// in the output rows (path 8), which it cannot do in place; callers that call
// in place and cannot allocate device memory at all (code under an allocator
// a host framework owns exclusively, real-time loops, processes that must not
// grow their device footprint) get softmax_fwd_noalloc: its scratch is the
// array below, which every GPU that loads this library holds from load until
// process exit.
#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

// The scratch of every softmax_fwd_noalloc call on this device: one (s, l)
// state per (row, chunk).  Its size is the hard limit on rows * chunks.
static __device__ __align__(256) float2 g_noalloc_states[kNoAllocMaxStates];

namespace {

// Device address of g_noalloc_states in the current device's context.  In
// host code the array's name is only a host-side stand-in, so the address
// comes from cudaGetSymbolAddress, looked up on every call (so that a context
// re-created after cudaDeviceReset is never handed a stale address).
cudaError_t states_address(float2 **ptr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_states);
    if (e != cudaSuccess) return e;
    *ptr = static_cast<float2 *>(p);
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
    float2 *states = nullptr;
    const cudaError_t e = states_address(&states);
    if (e != cudaSuccess) return e;
    switch (a.dtype) {
        case 0: return go<float>(a, chunks, chunk_vecs, grid, states);
        case 1: return go<__half>(a, chunks, chunk_vecs, grid, states);
        case 2: return go<__nv_bfloat16>(a, chunks, chunk_vecs, grid, states);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mbrs
