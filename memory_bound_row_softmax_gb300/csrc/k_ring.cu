// k_ring.cu -- path 5 instantiations: persistent blocks or clusters fed by a
// ring of TMA bulk copies.  The grid is one wave of co-resident blocks
// (clusters), sized with the occupancy API and cached per device and shape.
#include <atomic>
#include <mutex>
#include <vector>

#include "kernels.cuh"
#include "launch.h"

namespace mbrs {

namespace {
constexpr int kMaxDevices = 64;

template <typename T, int THREADS, int VPT, bool CL>
cudaError_t prepare(int device) {
    static std::atomic<unsigned long long> done{0};
    const unsigned long long bit = 1ull << (device & (kMaxDevices - 1));
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    auto fn = k_ring_rows<T, THREADS, VPT, CL>;
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

struct GridKey {
    int device;
    const void *fn;
    int csize;
    int64_t smem;
    int64_t per_wave;  // co-resident blocks (csize 1) or clusters (csize > 1) on the whole GPU
};

// Co-resident blocks (or clusters) of this kernel on the current device.
template <typename T, int THREADS, int VPT, bool CL>
cudaError_t per_wave(int device, int csize, int64_t smem, int64_t *out) {
    static std::mutex mu;
    static std::vector<GridKey> cache;
    const void *fn = reinterpret_cast<const void *>(k_ring_rows<T, THREADS, VPT, CL>);
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const auto &k : cache)
            if (k.device == device && k.fn == fn && k.csize == csize && k.smem == smem) {
                *out = k.per_wave;
                return cudaSuccess;
            }
    }
    int64_t n = 0;
    if (csize == 1) {
        int per_sm = 0, sms = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_ring_rows<T, THREADS, VPT, CL>,
                                                                      THREADS, (size_t)smem);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
        if (e != cudaSuccess) return e;
        n = (int64_t)per_sm * sms;
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)csize, 1, 1);
        cfg.blockDim = dim3(THREADS, 1, 1);
        cfg.dynamicSmemBytes = (size_t)smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)csize;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, k_ring_rows<T, THREADS, VPT, CL>, &cfg);
        if (e != cudaSuccess) return e;
        n = clusters;
    }
    if (n < 1) return cudaErrorInvalidConfiguration;
    std::lock_guard<std::mutex> lock(mu);
    cache.push_back({device, fn, csize, smem, n});
    *out = n;
    return cudaSuccess;
}

int sms_of(int device) {
    int sms = 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    return sms > 0 ? sms : 1;
}

// Persistent units (blocks, or clusters) for `rows` rows given that at most
// `wave` fit at once.  Each unit walks ceil(rows / U) rows and the call lasts
// about as long as its busiest unit, so take the U in [wave/2, wave] with the
// least ceil(rows/U) * U (the most even split), the larger on ties.  Single
// blocks are counted in whole SMs (`step` = SMs) so every SM gets as many.
int64_t balanced_units(int64_t rows, int64_t wave, int64_t step) {
    if (rows <= wave) return rows;
    int64_t best = wave, best_cost = INT64_MAX;
    const int64_t lo = std::max<int64_t>(step, wave / 2);
    for (int64_t u = (wave / step) * step; u >= lo; u -= step) {
        const int64_t cost = ((rows + u - 1) / u) * u;
        if (cost < best_cost) {
            best_cost = cost;
            best = u;
        }
    }
    return best;
}

template <typename T, int THREADS, int VPT, bool CL>
cudaError_t go(const LaunchArgs &a, const RingCfg &c, int64_t wait_ns, int starve, int64_t *grid_out) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e == cudaSuccess) e = prepare<T, THREADS, VPT, CL>(device);
    int64_t wave = 0;
    if (e == cudaSuccess) e = per_wave<T, THREADS, VPT, CL>(device, c.csize, c.smem, &wave);
    if (e != cudaSuccess) return e;
    // single blocks: an even split of rows over whole SMs; clusters: the full
    // wave, so that their blocks sit evenly on the SMs
    const int64_t units = c.csize == 1 ? balanced_units(a.rows, wave, sms_of(device)) : std::min(a.rows, wave);
    const int64_t grid = units * c.csize;
    if (grid_out) *grid_out = grid;
    if (!a.in) return cudaSuccess;  // grid query only
    return launch_kernel(k_ring_rows<T, THREADS, VPT, CL>, a, grid, THREADS, (size_t)c.smem, c.csize > 1 ? c.csize : 0,
                         static_cast<const T *>(a.in), static_cast<T *>(a.out), a.rows, a.cols, a.stride, c.stages,
                         c.slice_vecs, wait_ns, starve);
}

template <typename T, int THREADS>
cudaError_t by_vpt(const LaunchArgs &a, const RingCfg &c, int64_t w, int s, int64_t *g) {
    if (c.csize > 1) {  // cluster rings: 256..1024 threads, 2 or 4 vectors each
        if constexpr (THREADS >= 256) {
            if (c.vpt == 2) return go<T, THREADS, 2, true>(a, c, w, s, g);
            if (c.vpt == 4) return go<T, THREADS, 4, true>(a, c, w, s, g);
        }
        return cudaErrorInvalidValue;
    }
    switch (c.vpt) {
        case 1: return go<T, THREADS, 1, false>(a, c, w, s, g);
        case 2: return go<T, THREADS, 2, false>(a, c, w, s, g);
        case 4: return go<T, THREADS, 4, false>(a, c, w, s, g);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t by_shape(const LaunchArgs &a, const RingCfg &c, int64_t w, int s, int64_t *g) {
    switch (c.threads) {
        case 64: return by_vpt<T, 64>(a, c, w, s, g);
        case 128: return by_vpt<T, 128>(a, c, w, s, g);
        case 256: return by_vpt<T, 256>(a, c, w, s, g);
        case 512: return by_vpt<T, 512>(a, c, w, s, g);
        case 1024: return by_vpt<T, 1024>(a, c, w, s, g);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

bool ring_shape_ok(int threads, int vpt, int csize) {
    const bool t = threads == 64 || threads == 128 || threads == 256 || threads == 512 || threads == 1024;
    if (csize > 1) return threads >= 256 && t && (vpt == 2 || vpt == 4);
    return t && (vpt == 1 || vpt == 2 || vpt == 4);
}

int64_t ring_smem_bytes(int stages, int slice_vecs, int threads) {
    return RingLayout(stages, slice_vecs, threads).bytes;
}

cudaError_t launch_ring(const LaunchArgs &a, const RingCfg &c, int64_t wait_ns, int starve, int64_t *grid) {
    if (c.csize < 1 || c.csize > kMaxCluster || c.stages < 1) return cudaErrorInvalidValue;
    switch (a.dtype) {
        case 0: return by_shape<float>(a, c, wait_ns, starve, grid);
        case 1: return by_shape<__half>(a, c, wait_ns, starve, grid);
        case 2: return by_shape<__nv_bfloat16>(a, c, wait_ns, starve, grid);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_clear_ring_error_word(unsigned int *word) {
    cudaError_t e = cudaMemcpyFromSymbol(word, g_error_word, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(unsigned int), 0, cudaMemcpyHostToDevice);
}

}  // namespace mbrs
