// launch.h -- host-side interface between the C ABI (abi.cu) and the per-path
// translation units that hold the kernel instantiations.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

namespace mbrs {

// softmax_fwd_masked: row r keeps columns c < kept(r) = clamp((r mod period)
// + off + 1, 0, cols) (period 0: r itself), and its scores are x * scale,
// entered into the exponent as k = scale * log2 e.
struct CausalMask {
    int64_t off = 0, period = 0;
    float k = 1.4426950408889634f;  // log2 e: scale 1
    __host__ __device__ int64_t kept(int64_t row, int64_t cols) const {
        // 32-bit remainder when both fit (a 64-bit one is a long instruction sequence)
        const bool narrow = row <= 0x7fffffff && period <= 0x7fffffff;
        const int64_t q = period <= 0 ? row
                          : narrow   ? (int64_t)((uint32_t)row % (uint32_t)period)
                                     : row % period;
        const int64_t n = q + off + 1;
        return n < 0 ? 0 : (n > cols ? cols : n);
    }
};

struct LaunchArgs {
    const void *in;
    void *out;
    int64_t rows, cols, stride;
    int dtype;      // 0 f32, 1 f16, 2 bf16
    int vec_store;  // out shares in's 16-byte phase
    cudaStream_t stream;
    int overlap;    // launch with programmatic stream serialisation
    int whole;      // every row is whole 16-byte vectors: in and out 16-byte
                    // aligned, row stride and width multiples of 16 bytes
    CausalMask mask;  // masked launches only
};

// Device error word bits (k_cluster.cu holds the word): a bounded wait ran
// out; a cluster kernel found itself launched without a cluster (it then
// returns before any cluster access).
constexpr unsigned int kErrWaitTimeout = 1u;
constexpr unsigned int kErrNotCluster = 2u;

// Kernel variants of the warp and block paths.
constexpr int kPlainRows = 0, kWholeRows = 1, kMaskedRows = 2, kMaskedWholeRows = 3;

// Launch `kernel` on a.stream; csize >= 1 makes it a cluster launch with
// clusters of csize blocks (kernels that use cluster instructions need it,
// even for csize == 1), csize == 0 a plain launch.
// With a.overlap set the launch allows programmatic dependent launch: the
// grid may be scheduled while the previous kernel in the stream is still
// finishing, so that its launch latency and block rasterisation overlap that
// kernel's tail.  Every kernel of this library therefore starts with
// griddepcontrol.wait (pdl_enter), which returns only once the previous grid
// has completed and its memory operations are visible, before its first
// global-memory access.
template <typename... P, typename... A>
cudaError_t launch_kernel(void (*kernel)(P...), const LaunchArgs &a, int64_t grid, int threads, size_t smem,
                          int csize, A &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (csize >= 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)csize;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (a.overlap) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<A &&>(args)...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Each launcher returns cudaErrorInvalidValue when no instantiation matches
// the requested shape (the planner only asks for shapes that exist).
bool warp_shape_ok(int group, int vpt);
cudaError_t launch_warp(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid);

bool cta_shape_ok(int threads, int vpt);
cudaError_t launch_cta(const LaunchArgs &a, int threads, int vpt, int64_t grid);
// the instantiations for a.whole (k_warp_whole.cu, k_cta_whole.cu)
cudaError_t launch_warp_whole(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid);
cudaError_t launch_cta_whole(const LaunchArgs &a, int threads, int vpt, int64_t grid);
// scaled, causally masked rows with a.mask (k_masked_warp.cu, k_masked.cu):
// the warp and block shapes of paths 1 and 2, and the streaming cluster
cudaError_t launch_warp_masked(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid);
cudaError_t launch_cta_masked(const LaunchArgs &a, int threads, int vpt, int64_t grid);
// ... their a.whole instantiations (k_masked_warp_whole.cu, k_masked_whole.cu)
cudaError_t launch_warp_masked_whole(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid);
cudaError_t launch_cta_masked_whole(const LaunchArgs &a, int threads, int vpt, int64_t grid);
cudaError_t launch_stream_masked(const LaunchArgs &a, int threads, int vpt, int csize, int64_t wait_ns,
                                 int starve);

// path 3: 16-bit rows, slices of threads x 8 vectors held in registers
// (threads 256 or 512).  starve != 0 (a test hook of every cluster kernel)
// makes the state exchange send nothing, so its bounded waits run out.
bool cluster_shape_ok(int threads, int vpt, int elem_bytes);
int64_t cluster_smem_bytes(int threads);
cudaError_t launch_cluster(const LaunchArgs &a, int threads, int vpt, int csize, int64_t wait_ns, int starve);
// path 7: narrow dense rows (stride == cols) staged through shared memory
// rows_per_span at a time, one thread per row, kPackedThreads per block
constexpr int kPackedThreads = 128;
constexpr int64_t kPackedMaxSmem = 48 * 1024;
int64_t packed_smem_bytes(int64_t rows_per_span, int64_t cols, int elem_bytes);
cudaError_t launch_packed(const LaunchArgs &a, int rows_per_span, int64_t grid);

// path 6: a cluster of csize blocks per row streaming slices of any length
// twice (pass 1 states, cluster exchange, pass 2 re-read and write)
bool stream_shape_ok(int threads, int vpt);
int64_t stream_smem_bytes(int threads);
cudaError_t launch_stream(const LaunchArgs &a, int threads, int vpt, int csize, int64_t wait_ns, int starve);
// read this device's error word after synchronising `stream`, then clear it
cudaError_t read_clear_error_word(cudaStream_t stream, unsigned int *word);

// path 8: a few very long rows over the whole grid, their per-chunk states in
// the output row itself (k_grid.cu): two launches of `threads` threads x `vpt`
// vectors (grid_shape_ok; kGridThreads x kGridVpt by default); a.in must
// differ from a.out; `chunks` slots of 8 bytes and a 4-byte counter, from the
// row's first 4-byte aligned byte, must fit in the row (8 chunks + 8 <= row
// bytes)
constexpr int kGridThreads = 512, kGridVpt = 4;

// softmax_masked_copy (k_pattern_copy.cu): a.mask's kept entries of each row
// copied, the rest zero-filled; rows of whole 16-byte vectors (a.whole).
cudaError_t launch_masked_copy(const LaunchArgs &a, int threads, int64_t grid);
bool grid_shape_ok(int threads, int vpt);
cudaError_t launch_grid(const LaunchArgs &a, int threads, int vpt, int64_t chunks, int64_t chunk_vecs,
                        int64_t grid);

// softmax_fwd_noalloc: the split path with its per-chunk states in a fixed
// device array of kNoAllocMaxStates float2 (k_noalloc.cu); rows * chunks must
// not exceed it.  Launch shape: 256 threads, 4 vectors per thread.
constexpr int64_t kNoAllocMaxStates = 65536;
constexpr int kNoAllocThreads = 256, kNoAllocVpt = 4;
cudaError_t launch_split_noalloc(const LaunchArgs &a, int64_t chunks, int64_t chunk_vecs, int64_t grid);

// host state of the softmax ABI that the attention ABI (attention_abi.cu)
// shares: the device's SM count (cached) and the bounded-wait limit
int host_device_sms(int *sms);
int64_t host_wait_ns();

}  // namespace mbrs
