// launch.h -- host-side interface between the C ABI (abi.cu) and the per-path
// translation units that hold the kernel instantiations.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

namespace mbrs {

struct LaunchArgs {
    const void *in;
    void *out;
    int64_t rows, cols, stride;
    int dtype;      // 0 f32, 1 f16, 2 bf16
    int vec_store;  // out shares in's 16-byte phase
    cudaStream_t stream;
};

// Each launcher returns cudaErrorInvalidValue when no instantiation matches
// the requested shape (the planner only asks for shapes that exist).
bool warp_shape_ok(int group, int vpt);
cudaError_t launch_warp(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid);

bool cta_shape_ok(int threads, int vpt);
cudaError_t launch_cta(const LaunchArgs &a, int threads, int vpt, int64_t grid);

bool cluster_shape_ok(int threads, int vpt, int elem_bytes);
int64_t cluster_smem_bytes(int threads, int vpt);
cudaError_t launch_cluster(const LaunchArgs &a, int threads, int vpt, int csize, int64_t wait_ns, int starve);
// read this device's error word after synchronising `stream`, then clear it
cudaError_t read_clear_error_word(cudaStream_t stream, unsigned int *word);

// path 5: persistent TMA ring.  grid (out) is the persistent grid actually
// used; with a.in == nullptr nothing is launched (grid query only).
struct RingCfg {
    int threads, vpt, csize, stages, slice_vecs;
    int64_t smem;
};
bool ring_shape_ok(int threads, int vpt, int csize);
int64_t ring_smem_bytes(int stages, int slice_vecs, int threads);
cudaError_t launch_ring(const LaunchArgs &a, const RingCfg &c, int64_t wait_ns, int starve, int64_t *grid);
// read this translation unit's device error word (after a stream sync), then clear it
cudaError_t read_clear_ring_error_word(unsigned int *word);

// softmax_fwd_noalloc: the split path with its per-chunk states in a fixed
// device array of kNoAllocMaxStates float2 (k_noalloc.cu); rows * chunks must
// not exceed it.  Launch shape: 256 threads, 4 vectors per thread.
constexpr int64_t kNoAllocMaxStates = 65536;
constexpr int kNoAllocThreads = 256, kNoAllocVpt = 4;
cudaError_t launch_split_noalloc(const LaunchArgs &a, int64_t chunks, int64_t chunk_vecs, int64_t grid);

bool split_shape_ok(int threads, int vpt);
cudaError_t launch_split(const LaunchArgs &a, int threads, int vpt, int64_t chunks, int64_t chunk_vecs,
                         int64_t grid, void *scratch);

}  // namespace mbrs
