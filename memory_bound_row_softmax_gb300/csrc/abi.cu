// abi.cu -- the C ABI: argument checks, the width-based dispatcher, launch
// planning and the diagnostics declared in include/mbrs_softmax.h.
//
// Dispatch (page "fused-softmax-roofline", section on the shapes where the
// fused kernel loses: the fixed per-row costs must be paid per lane group, not
// per block, for short rows; page "GPU Kernels - Implementing and optimizing
// Softmax", sections "CUDA optimized for block per row" and "CUDA scaling
// threads": wide rows need more threads per row so that enough loads are in
// flight):
//   narrow dense rows off the 16-byte grid  path 7, staged through shared memory
//   rows a warp's registers hold            path 1, 2..32 lanes per row
//   16-bit rows a cluster's registers hold  path 3, a cluster per row
//   other rows a block's registers hold     path 2, a block per row
//   a few very long rows, out != in         path 8, chunks over the whole grid,
//                                           states in the output rows
//   longer rows                             path 6, a cluster per row streaming
//                                           its slices twice
// Every path keeps its partial states on chip -- path 8 in the output rows it
// is about to overwrite: no call allocates memory.
#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "mbrs_softmax.h"
#include "attention_launch.h"
#include "launch.h"

using namespace mbrs;

namespace {

constexpr int kAbiVersion = 20200;  // 2.2.0
constexpr int kVecBytes = 16;
constexpr int kMaxDevices = 64;
constexpr int64_t kDefaultWaitNs = 1000000000;  // 1 s
constexpr int64_t kMaxGrid = 0x7fffffff;
constexpr int64_t kGridMinRowBytes = 1 << 20;  // path 8 only for rows this long

std::atomic<int> g_last_path{0};
std::atomic<int> g_force_path{0}, g_force_threads{0}, g_force_vpt{0}, g_force_group{0};
std::atomic<int64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_starve{0};
std::atomic<int> g_overlap{1};

struct Plan {
    int path = 0, threads = 0, vpt = 0, group = 1, launches = 0, vec_store = 0, whole = 0;
    int64_t grid = 0, smem = 0, hbm = 0, chunks = 0, chunk_vecs = 0;
};

// A launch shape asked for: path 0 = automatic; threads / vpt / group 0 =
// the planner's own choice for that path.
struct Shape {
    int path = 0, threads = 0, vpt = 0, group = 0;
};

Shape forced_shape() {
    return Shape{g_force_path.load(), g_force_threads.load(), g_force_vpt.load(), g_force_group.load()};
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int next_pow2(int64_t v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Shape of the block-per-row register kernel.  For each thread count (a power
// of two) the row needs vpt = ceil(nv / threads) vectors per thread, rounded
// up to an instantiated count (2..6, 8, 10; at most 5 with 1024 threads).
// Registers per thread: 4 per vector plus ~24, or the 64 the kernel is bounded
// to from 6 vectors up.  The shape kept is the one with the most row bytes
// resident per SM (rows per SM by threads and registers, times the row),
// ties going to fewer threads -- measured, wide rows run best with 256 threads
// x 8 vectors (8192-wide fp32: 59 us, against 68 us for 512 x 4).
int cta_vpt_round(int64_t v) {
    if (v <= 2) return 2;
    if (v <= 6) return (int)v;
    return v <= 8 ? 8 : 10;
}
int64_t cta_rows_per_sm(int threads, int vpt) {
    const int64_t regs = vpt >= 6 ? 64 : 4 * vpt + 24;
    return std::min<int64_t>(std::min<int64_t>(2048 / threads, 65536 / (threads * regs)), 32);
}
bool cta_shape(int64_t nv, int *threads_out, int *vpt_out) {
    int64_t best = -1;
    for (int threads = 64; threads <= 1024; threads *= 2) {
        const int64_t need = cdiv(nv, threads);
        if (need > (threads == 1024 ? 5 : 10)) continue;
        // 64 or 128 threads x 9-10 vectors lose to twice the threads x 5
        // (2055-wide fp32: 58.1 us on 64 x 10, 56.3 on 128 x 5; 4103-wide:
        // 58.3 on 128 x 10, 56.5 on 256 x 5; from 256 threads they tie)
        if (threads < 256 && need > 8) continue;
        const int vpt = cta_vpt_round(need);
        const int64_t resident = cta_rows_per_sm(threads, vpt);
        if (resident > best) {
            best = resident;
            *threads_out = threads;
            *vpt_out = vpt;
        }
    }
    return best > 0;
}

int elem_bytes(int dtype) { return dtype == SOFTMAX_F32 ? 4 : 2; }

// Host-side argument checks, in the order the header documents.
int check_args(uint64_t in, uint64_t out, int64_t rows, int64_t cols, int64_t row_stride, int dtype,
               int64_t *extent_bytes) {
    if (dtype != SOFTMAX_F32 && dtype != SOFTMAX_F16 && dtype != SOFTMAX_BF16) return SOFTMAX_ERR_DTYPE;
    if (rows < 0 || cols < 1) return SOFTMAX_ERR_SHAPE;
    if (row_stride < cols) return SOFTMAX_ERR_STRIDE;
    const int es = elem_bytes(dtype);
    // extent = (rows - 1) * row_stride + cols elements must fit in int64 bytes
    if (rows > 0) {
        if (rows - 1 > (INT64_MAX - cols) / row_stride) return SOFTMAX_ERR_SHAPE;
        const int64_t ext = (rows - 1) * row_stride + cols;
        if (ext > INT64_MAX / es) return SOFTMAX_ERR_SHAPE;
        *extent_bytes = ext * es;
    } else {
        *extent_bytes = 0;
        return SOFTMAX_OK;
    }
    if (in == 0 || out == 0) return SOFTMAX_ERR_NULL;
    if (in % es != 0 || out % es != 0) return SOFTMAX_ERR_ALIGN;
    if (in != out) {
        const uint64_t n = (uint64_t)*extent_bytes;
        const bool disjoint = (in + n <= out) || (out + n <= in);
        if (!disjoint) return SOFTMAX_ERR_OVERLAP;
    }
    return SOFTMAX_OK;
}

int device_sms(int *sms) {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SOFTMAX_ERR_CUDA;
    const int slot = dev & (kMaxDevices - 1);
    int v = cache[slot].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SOFTMAX_ERR_CUDA;
        cache[slot].store(v, std::memory_order_relaxed);
    }
    *sms = v;
    return SOFTMAX_OK;
}

// The launch for one call.  nv bounds the vectors any row needs: rows whose
// byte stride is a multiple of 16 share the first row's phase; otherwise a row
// may start up to V-1 elements into its first vector.
int make_plan(uint64_t in, uint64_t out, int64_t rows, int64_t cols, int64_t row_stride, int dtype, int sms,
              const Shape &force, Plan *p) {
    const int es = elem_bytes(dtype), V = kVecBytes / es;
    const bool uniform = ((row_stride * es) % kVecBytes) == 0;
    const int64_t head = (int64_t)((in % kVecBytes) / es);
    const int64_t nv = uniform ? cdiv(head + cols, V) : cdiv(cols + V - 1, V);
    p->vec_store = (in % kVecBytes) == (out % kVecBytes);
    // every row made of whole 16-byte vectors: the kernels' edge-free variants
    p->whole = in % kVecBytes == 0 && out % kVecBytes == 0 && (row_stride * es) % kVecBytes == 0 &&
               (cols * es) % kVecBytes == 0;
    p->hbm = 2 * rows * cols * es;

    const int fpath = force.path, fth = force.threads, fvpt = force.vpt, fgrp = force.group;
    int path = fpath;
    if (path == SOFTMAX_PATH_AUTO) {
        if (row_stride == cols && (cols * es) % kVecBytes != 0 && p->vec_store && cols <= 48) {
            // narrow dense rows off the 16-byte grid: staged through shared
            // memory, one thread per row (fp32 1282051 x 39: 64.7 us, a warp
            // path lane group per row 81.5; 400000 x 7: 6.7 against 15.0;
            // 71 wide it loses, 77.8 against 58.9)
            path = SOFTMAX_PATH_PACKED;
        } else if (nv <= 32 * 9 && (cols <= 1024 || p->whole || es == 2)) {
            // a warp per row while a warp's registers hold it; past 1024
            // columns for rows of whole vectors and for 16-bit rows, whose
            // partial end vectors take a few aligned partial stores (4096 x
            // 2048 fp16: warp 5.8 us, block 6.3 us; 8192 x 2055 fp16: warp
            // 11.6 us, block 13.4; 16384 x 2049 bf16: 21.4 against 24.5).
            // Ragged fp32 rows stay on the block path (their edges go element
            // by element)
            path = SOFTMAX_PATH_WARP;
        } else if (nv > 512 * 10 && es == 2 && cdiv(nv, 2048) <= 16 && rows * cdiv(nv, 2048) >= sms) {
            // 16-bit rows longer than a block's registers: a cluster holding the
            // row in registers, 2048 vectors per block (c5: 52 us, ring 57 us)
            path = SOFTMAX_PATH_CLUSTER;
        } else if (nv <= 512 * 10) {
            // a block per row while its registers hold the row: it beats the
            // ring at every such width measured (8192 x 2816 fp16: block 14.4
            // us, ring 17.1; 4096 x 2816 fp32: 14.0 against 19.5)
            path = SOFTMAX_PATH_CTA;
        } else if (rows * 16 < sms && in != out && cols * es >= kGridMinRowBytes) {
            // a few rows of 1 MiB or more: no cluster can spread them over
            // more than 16 SMs each, so their chunks go over the whole grid,
            // their states meeting in the output rows (fp32 1 x 4e6: 34.8 us
            // on the streaming cluster, 10.9 here)
            path = SOFTMAX_PATH_GRID;
        } else {
            // longer rows: a cluster streaming its slices twice, about one
            // 1024-vector tile per block.  Measured against a TMA-fed ring and
            // a TMA-staged cluster it won at every long width tried
            // (1525 x 32768 fp32: 58.8 us, ring 62.5, TMA cluster 64.2;
            // 381 x 131072: 60.4, ring 74.0; 300 x 40000: 18.7, ring 25.0).
            // Also for a few long rows (rows * 16 < SMs) in place or under
            // 1 MiB, which path 8 does not take (bf16 9 x 262144: 4.7 us
            // here, 7.2 on path 8)
            path = SOFTMAX_PATH_STREAM;
        }
    }
    p->path = path;
    p->launches = 1;
    switch (path) {
        case SOFTMAX_PATH_WARP: {
            int g, vpt;
            if (fgrp > 0) {
                g = fgrp;
                vpt = fvpt > 0 ? fvpt : (int)cdiv(nv, g);
            } else {
                // lanes per row: the group (2..32 lanes, up to 8 vectors each; 9
                // for a whole warp) with the most row bytes resident per SM --
                // warps per SM by registers (4 per vector + ~24) times rows per warp
                int64_t best = -1;
                g = 32;
                vpt = (int)cdiv(nv, 32);
                // (measured: sub-warp groups with 6+ vectors per lane lose -- a
                // 39-wide fp32 row ran 70 us on 2 x 6 against 62 us on 4 x 3)
                for (int gg = 2; gg <= 32; gg *= 2) {
                    const int64_t v = cdiv(nv, gg);
                    if (v > (gg == 32 ? 9 : 5)) continue;
                    const int64_t warps = std::min<int64_t>(64, 65536 / (32 * (4 * v + 24)));
                    const int64_t resident = warps * (32 / gg);
                    if (resident > best) {
                        best = resident;
                        g = gg;
                        vpt = (int)v;
                    }
                }
                if (fvpt > 0) vpt = fvpt;
            }
            if (!warp_shape_ok(g, vpt) || (int64_t)g * vpt < nv) return SOFTMAX_ERR_UNSUPPORTED;
            // 8 rows per block for rows of 6+ vectors per lane (4096 x 2048
            // fp16: 5.8 us at 256 threads, 6.0 us at 128), else 4
            int threads = fth > 0 ? fth : (g == 32 && vpt >= 6 ? 256 : 128);
            if (fth <= 0)  // spread small problems over more SMs
                while (threads > 32 && cdiv(rows * g, threads) < sms) threads /= 2;
            if (fth <= 0 && cdiv(rows * g, threads) >= sms) {
                // One wave of blocks: the SM with the most blocks sets the time,
                // so take the block size (down to half, in whole warps) that
                // gives the fewest rows to the busiest SM (fp16 4096 x 2048:
                // 8 rows per block put 32 rows on some SMs, 5.53 us; 7 rows,
                // 28 at most, 5.37 us).  Several waves balance themselves.
                const int64_t regs = 4 * vpt + 24;
                int best_t = threads;
                int64_t best_load = INT64_MAX;
                for (int t = threads; t >= std::max(32, threads / 2); t -= 32) {
                    if (t % g != 0) continue;
                    const int64_t rpb = t / g, blocks = cdiv(rows, rpb);
                    const int64_t per_sm = std::min<int64_t>({32, 2048 / t, 65536 / (t * regs)});
                    const int64_t load = blocks <= per_sm * sms ? cdiv(blocks, sms) * rpb : cdiv(rows, sms);
                    if (load < best_load) {
                        best_load = load;
                        best_t = t;
                    }
                }
                threads = best_t;
            }
            if (threads < 32 || threads > 256 || threads % 32 != 0 || threads % g != 0)
                return SOFTMAX_ERR_UNSUPPORTED;
            p->threads = threads;
            p->vpt = vpt;
            p->group = g;
            p->grid = std::min<int64_t>(cdiv(rows * g, threads), kMaxGrid);
            break;
        }
        case SOFTMAX_PATH_CTA: {
            // the fewest threads (a power of two) that need at most 4 vectors each
            // (5 at 1024 threads); vpt = what the row then needs, not a rounded-up 4
            int threads = fth, vpt = fvpt;
            if (threads <= 0) {
                int v = 0;
                threads = 1024;
                cta_shape(nv, &threads, &v);
                if (vpt <= 0) vpt = v;
            }
            if (vpt <= 0) vpt = cta_vpt_round(cdiv(nv, threads));
            if (!cta_shape_ok(threads, vpt) || (int64_t)threads * vpt < nv) return SOFTMAX_ERR_UNSUPPORTED;
            p->threads = threads;
            p->vpt = vpt;
            p->grid = std::min(rows, kMaxGrid);
            break;
        }
        case SOFTMAX_PATH_CLUSTER: {
            // 16-bit rows: slices of 256 (or 512) threads x 8 vectors held in
            // registers, as many blocks as the row needs (fp32 rows would
            // spill there)
            const int threads = fth > 0 ? fth : (cdiv(nv, 256 * 8) <= 16 ? 256 : 512);
            const int vpt = fvpt > 0 ? fvpt : 8;
            const int64_t csize = fgrp > 0 ? fgrp : cdiv(nv, (int64_t)threads * vpt);
            if (!cluster_shape_ok(threads, vpt, es) || csize < 1 || csize > 16) return SOFTMAX_ERR_UNSUPPORTED;
            if (cdiv(nv, csize) > (int64_t)threads * vpt) return SOFTMAX_ERR_UNSUPPORTED;
            if (rows * csize > kMaxGrid) return SOFTMAX_ERR_UNSUPPORTED;
            p->threads = threads;
            p->vpt = vpt;
            p->group = (int)csize;
            p->grid = rows * csize;
            p->smem = cluster_smem_bytes(threads);
            break;
        }
        case SOFTMAX_PATH_PACKED: {
            // one thread per row, 128 rows (times vpt, 1 unless forced: more
            // rows per span measured slower) per staged span
            if (row_stride != cols || !p->vec_store || (fgrp > 0 && fgrp != 1)) return SOFTMAX_ERR_UNSUPPORTED;
            const int64_t k = fvpt > 0 ? fvpt : 1;
            const int64_t rps = (int64_t)kPackedThreads * k;
            if (rps > 0x7fffffff || packed_smem_bytes(rps, cols, es) > kPackedMaxSmem) return SOFTMAX_ERR_UNSUPPORTED;
            p->threads = kPackedThreads;
            p->vpt = (int)k;
            p->group = 1;
            p->grid = std::min<int64_t>(cdiv(rows, rps), kMaxGrid);
            p->smem = packed_smem_bytes(rps, cols, es);
            break;
        }
        case SOFTMAX_PATH_STREAM: {
            // 4 vectors per thread; 256 threads per block, or more while 16
            // blocks would need more than two tiles each; then as many blocks
            // (<= 16) as give about one tile each.  Measured: 1525 x 32768 fp32
            // 58.8 us on 8 x (256 x 4); 190 x 262144 64.2 us on 16 x (512 x 4)
            // (78.6 on 256); 64 x 2^20 105.6 us on 16 x (1024 x 4) (139 on 256).
            // With too few rows to give every SM a block (rows * 16 < SMs) a
            // block's bytes in flight bound the time, so the blocks grow to one
            // tile per block, up to 1024 threads (bf16 9 x 262144: 4.7 us on
            // 512 threads, 5.5 on 256; fp32 3 x 10^6: 12.3 on 1024, 14.5 on 512)
            const int vpt = fvpt > 0 ? fvpt : 4;
            int threads = fth;
            if (threads <= 0) {
                threads = 256;
                if (rows * 16 < sms) {
                    while (threads < 1024 && cdiv(nv, 16 * (int64_t)vpt) > threads) threads *= 2;
                } else {
                    while (threads < 1024 && cdiv(nv, 16 * (int64_t)threads * vpt) > 2) threads *= 2;
                }
            }
            const int64_t csize =
                fgrp > 0 ? fgrp : std::min<int64_t>(16, std::max<int64_t>(1, cdiv(nv, (int64_t)threads * vpt)));
            if (!stream_shape_ok(threads, vpt) || csize < 1 || csize > 16 || rows * csize > kMaxGrid)
                return SOFTMAX_ERR_UNSUPPORTED;
            p->threads = threads;
            p->vpt = vpt;
            p->group = (int)csize;
            p->grid = rows * csize;
            p->smem = stream_smem_bytes(threads);
            p->hbm = 3 * rows * cols * es;
            break;
        }
        case SOFTMAX_PATH_GRID: {
            // about two 512-thread blocks per SM over all rows, the row cut
            // into that many equal chunks, the last taking the rest (forced:
            // up to `group` chunks of 3 vectors or more).  Measured on one
            // GB300 (us): fp32 1 x 4e6 10.9 (256-thread blocks, four per SM:
            // 12.3; 1024 x 4, one per SM: 11.7); fp32 3 x 1e6 9.7 (12.3);
            // bf16 1 x 2^22 8.5 (9.4).  The row's state region (8 bytes per
            // chunk and a counter) must fit in the row.
            if (in == out || nv < 3) return SOFTMAX_ERR_UNSUPPORTED;
            const int th = fth > 0 ? fth : kGridThreads, vp = fvpt > 0 ? fvpt : kGridVpt;
            if (!grid_shape_ok(th, vp)) return SOFTMAX_ERR_UNSUPPORTED;
            const int64_t want = fgrp > 0 ? fgrp : std::max<int64_t>(1, 2 * (int64_t)sms / rows);
            const int64_t chunk_vecs = std::max<int64_t>(3, nv / want);
            const int64_t k = std::max<int64_t>(1, std::min<int64_t>(want, nv / chunk_vecs));
            if (8 * k + 8 > cols * es || rows > kMaxGrid / k) return SOFTMAX_ERR_UNSUPPORTED;
            p->threads = th;
            p->vpt = vp;
            p->group = (int)k;
            p->chunks = k;
            p->chunk_vecs = chunk_vecs;
            p->grid = std::min<int64_t>(rows * k, (int64_t)sms * (2048 / th));
            p->launches = 2;
            p->hbm = 3 * rows * cols * es;
            break;
        }
        default:
            return SOFTMAX_ERR_UNSUPPORTED;
    }
    return SOFTMAX_OK;
}

// The grid path counts the blocks of a row with a 32-bit atomic add on a word
// of `out`: fine in device or managed memory, and in host memory when the
// device performs atomics on host memory natively (a coherent CPU-GPU link).
bool grid_atomics_ok(const void *out) {
    int dev = 0, native = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&native, cudaDevAttrHostNativeAtomicSupported, dev) != cudaSuccess)
        return false;
    if (native) return true;
    cudaPointerAttributes pa;
    std::memset(&pa, 0, sizeof(pa));
    if (cudaPointerGetAttributes(&pa, out) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return pa.type == cudaMemoryTypeDevice || pa.type == cudaMemoryTypeManaged;
}

int run(const Plan &p, const LaunchArgs &a) {
    cudaError_t e = cudaSuccess;
    switch (p.path) {
        case SOFTMAX_PATH_WARP: e = launch_warp(a, p.threads, p.group, p.vpt, p.grid); break;
        case SOFTMAX_PATH_CTA: e = launch_cta(a, p.threads, p.vpt, p.grid); break;
        case SOFTMAX_PATH_CLUSTER:
            e = launch_cluster(a, p.threads, p.vpt, p.group, g_wait_ns.load(), g_starve.load());
            break;
        case SOFTMAX_PATH_STREAM:
            e = launch_stream(a, p.threads, p.vpt, p.group, g_wait_ns.load(), g_starve.load());
            break;
        case SOFTMAX_PATH_PACKED: e = launch_packed(a, kPackedThreads * p.vpt, p.grid); break;
        case SOFTMAX_PATH_GRID:
            if (!grid_atomics_ok(a.out)) return SOFTMAX_ERR_UNSUPPORTED;
            e = launch_grid(a, p.threads, p.vpt, p.chunks, p.chunk_vecs, p.grid);
            break;
        default: return SOFTMAX_ERR_UNSUPPORTED;
    }
    if (e == cudaErrorInvalidValue) return SOFTMAX_ERR_UNSUPPORTED;
    return e == cudaSuccess ? SOFTMAX_OK : SOFTMAX_ERR_CUDA;
}

// Split-path shape for softmax_fwd_noalloc: enough chunks to give every SM two
// blocks' worth of 256-thread blocks twice over, no chunk smaller than one
// tile, and chunks per row capped so that rows * chunks fits the fixed array.
int plan_noalloc(uint64_t in, int64_t rows, int64_t cols, int64_t row_stride, int dtype, int sms, int64_t *chunks,
                 int64_t *chunk_vecs, int64_t *grid) {
    if (rows > kNoAllocMaxStates) return SOFTMAX_ERR_SCRATCH_LIMIT;
    const int es = elem_bytes(dtype), V = kVecBytes / es;
    const bool uniform = ((row_stride * es) % kVecBytes) == 0;
    const int64_t head = (int64_t)((in % kVecBytes) / es);
    const int64_t nv = uniform ? cdiv(head + cols, V) : cdiv(cols + V - 1, V);
    const int64_t tile = (int64_t)kNoAllocThreads * kNoAllocVpt;
    const int64_t per_sm = 2048 / kNoAllocThreads;
    int64_t k = std::max<int64_t>(1, std::min(cdiv((int64_t)sms * per_sm * 2, rows), cdiv(nv, tile)));
    k = std::max<int64_t>(1, std::min(k, kNoAllocMaxStates / rows));
    const int64_t cv = cdiv(cdiv(nv, k), tile) * tile;
    *chunk_vecs = cv;
    *chunks = cdiv(nv, cv);
    *grid = std::min<int64_t>(rows * *chunks, (int64_t)sms * per_sm * 4);
    return SOFTMAX_OK;
}

// ---------------------------------------------------------------------------
// shape-keyed autotune (page "GPU Kernels - Implementing and optimizing
// Softmax", section "Autotuning": time the candidate launch configurations on
// the real shape, keep the fastest)
// ---------------------------------------------------------------------------
struct TuneKey {
    int device = 0, dtype = 0, in_phase = 0, out_phase = 0, rows_log2 = 0;
    bool in_place = false;  // tuning runs out of place; in-place calls never match
    int64_t cols = 0, row_stride = 0;
    bool operator==(const TuneKey &o) const {
        return device == o.device && dtype == o.dtype && in_phase == o.in_phase && out_phase == o.out_phase &&
               rows_log2 == o.rows_log2 && in_place == o.in_place && cols == o.cols && row_stride == o.row_stride;
    }
};

int floor_log2(int64_t v) {
    int r = 0;
    while (v > 1) {
        v >>= 1;
        ++r;
    }
    return r;
}

TuneKey tune_key(int device, uint64_t in, uint64_t out, int64_t rows, int64_t cols, int64_t row_stride, int dtype) {
    TuneKey k;
    k.device = device;
    k.dtype = dtype;
    k.in_phase = (int)(in % kVecBytes);
    k.out_phase = (int)(out % kVecBytes);
    k.rows_log2 = floor_log2(rows);
    k.in_place = in == out;
    k.cols = cols;
    k.row_stride = row_stride;
    return k;
}

std::mutex g_tune_mu;
std::vector<std::pair<TuneKey, Shape>> g_tuned;  // guarded by g_tune_mu
std::atomic<int> g_tuned_count{0};

void store_tuned(const TuneKey &k, const Shape &s) {
    std::lock_guard<std::mutex> lock(g_tune_mu);
    for (auto &e : g_tuned)
        if (e.first == k) {
            e.second = s;
            return;
        }
    g_tuned.emplace_back(k, s);
    g_tuned_count.store((int)g_tuned.size());
}

// The shape a call asks for: a forced one, else the tuned one for its key,
// else automatic.  No CUDA call while the cache is empty.
Shape call_shape(uint64_t in, uint64_t out, int64_t rows, int64_t cols, int64_t row_stride, int dtype) {
    const Shape f = forced_shape();
    if (f.path != SOFTMAX_PATH_AUTO || g_tuned_count.load() == 0) return f;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return f;
    const TuneKey k = tune_key(dev, in, out, rows, cols, row_stride, dtype);
    std::lock_guard<std::mutex> lock(g_tune_mu);
    for (const auto &e : g_tuned)
        if (e.first == k) return e.second;
    return f;
}

// The plan of a call: a forced shape, else the tuned one for its key, else
// the automatic choice.  A tuned shape this call cannot take (rows of another
// count in the same power-of-two bucket) gives way to the automatic choice.
int plan_call(uint64_t in, uint64_t out, int64_t rows, int64_t cols, int64_t row_stride, int dtype, int sms,
              Plan *p, Shape *used) {
    Shape want = call_shape(in, out, rows, cols, row_stride, dtype);
    int st = make_plan(in, out, rows, cols, row_stride, dtype, sms, want, p);
    if (st == SOFTMAX_ERR_UNSUPPORTED && want.path != SOFTMAX_PATH_AUTO && forced_shape().path == SOFTMAX_PATH_AUTO) {
        want = Shape{};
        st = make_plan(in, out, rows, cols, row_stride, dtype, sms, want, p);
    }
    if (used) *used = want;
    return st;
}

// Candidate shapes for rows of up to nv vectors: the automatic choice first,
// the shared-memory staged path for narrow dense rows, then every lane-group /
// block / cluster shape that can hold the row, the streaming cluster at
// three block sizes and, for rows longer than a block with out != in, the
// grid-wide path.
std::vector<Shape> tune_candidates(int64_t nv, int es, bool packed_ok, bool grid_ok) {
    std::vector<Shape> c;
    c.push_back(Shape{});
    if (packed_ok) c.push_back(Shape{SOFTMAX_PATH_PACKED, 0, 1, 0});
    if (nv <= 32 * 9)
        for (int g = 2; g <= 32; g *= 2) {
            const int64_t v = cdiv(nv, g);
            if (!warp_shape_ok(g, (int)v)) continue;
            for (int t = 64; t <= 256; t *= 2) c.push_back(Shape{SOFTMAX_PATH_WARP, t, (int)v, g});
        }
    if (nv <= 512 * 10)
        for (int t = 64; t <= 1024; t *= 2) {
            const int v = cta_vpt_round(cdiv(nv, t));
            if (cta_shape_ok(t, v) && (int64_t)t * v >= nv) c.push_back(Shape{SOFTMAX_PATH_CTA, t, v, 0});
        }
    if (nv > 512) {
        for (int t = 256; t <= 512; t *= 2)
            if (cluster_shape_ok(t, 8, es) && cdiv(nv, (int64_t)t * 8) <= 16)
                c.push_back(Shape{SOFTMAX_PATH_CLUSTER, t, 8, 0});
        for (int t = 256; t <= 1024; t *= 2) c.push_back(Shape{SOFTMAX_PATH_STREAM, t, 4, 0});
    }
    if (nv > 512 * 10 && grid_ok) c.push_back(Shape{SOFTMAX_PATH_GRID, 0, 0, 0});
    return c;
}

std::vector<Shape> candidates_for(uint64_t in, uint64_t out, int64_t cols, int64_t row_stride, int dtype) {
    const int es = elem_bytes(dtype), V = kVecBytes / es;
    const bool uniform = ((row_stride * es) % kVecBytes) == 0;
    const int64_t head = (int64_t)((in % kVecBytes) / es);
    const int64_t nv = uniform ? cdiv(head + cols, V) : cdiv(cols + V - 1, V);
    const bool packed_ok = row_stride == cols && (in % kVecBytes) == (out % kVecBytes) &&
                           packed_smem_bytes(kPackedThreads, cols, es) <= kPackedMaxSmem;
    return tune_candidates(nv, es, packed_ok, in != out);
}

void fill_public_plan(const Plan &p, softmax_plan_t *plan) {
    plan->path = p.path;
    plan->threads = p.threads;
    plan->vpt = p.vpt;
    plan->group = p.group;
    plan->launches = p.launches;
    plan->vec_store = p.vec_store;
    plan->grid = p.grid;
    plan->smem_bytes = p.smem;
    plan->scratch_bytes = 0;  // no path takes scratch
    plan->hbm_bytes = p.hbm;
    plan->whole_vectors = p.whole;
}

// ---------------------------------------------------------------------------
// host buffers (softmax_fwd_host): chunks of rows through three device slots,
// each slot with its own stream, so that a host-to-device copy, a softmax and
// a device-to-host copy of three chunks are in flight at once
// ---------------------------------------------------------------------------
constexpr int kHostSlots = 3;
// Default chunk: a quarter of the matrix, within 2 to 8 MiB (measured, fp16
// 4096 x 2048 through pinned memory: 1 MiB chunks 146 GB/s, 4 MiB 210,
// 64 MiB -- no overlap -- 179; fp32 4096 x 4096: 8 MiB 254, 1 MiB 154).
constexpr int64_t kHostChunkMin = 2 << 20, kHostChunkMax = 8 << 20;

struct HostPipe {
    std::mutex mu;  // held while a call queues its work
    bool ready = false;
    cudaStream_t s[kHostSlots] = {};
    cudaEvent_t start = nullptr;
    cudaEvent_t done[kHostSlots] = {};
};
HostPipe g_host_pipes[kMaxDevices];

// Create the pipe's streams and events (caller holds hp.mu).
cudaError_t host_pipe_ready(HostPipe &hp) {
    if (hp.ready) return cudaSuccess;
    cudaError_t e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming);
    for (int j = 0; j < kHostSlots && e == cudaSuccess; ++j) {
        e = cudaStreamCreateWithFlags(&hp.s[j], cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.done[j], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) hp.ready = true;
    return e;
}

// A slot holds n rows packed densely (row stride = cols: the host rows'
// padding is neither copied in nor out), starting 256-byte aligned.
int64_t host_slot_bytes(int64_t n, int64_t cols, int es) { return (n * cols * es + 255) / 256 * 256; }

// Rows per chunk: about chunk_bytes of row data, at least one, at most all.
int64_t host_chunk_rows(int64_t rows, int64_t cols, int es, int64_t chunk_bytes) {
    const int64_t cr = std::max<int64_t>(1, chunk_bytes / (cols * es));
    return std::min(cr, rows);
}

// Whether the current device can load and store the host range at `p`
// directly, at the same address: page-locked memory mapped into the unified
// address space (cudaHostAlloc, cudaHostRegister), device or managed memory,
// or pageable memory on a device that reaches it through the host's page
// tables (a coherent CPU-GPU link such as NVLink-C2C).  Nothing is launched
// when the answer is no.
int device_reaches(const void *p, bool *ok) {
    *ok = false;
    cudaPointerAttributes a;
    std::memset(&a, 0, sizeof(a));
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // unregistered memory on older runtimes: not sticky
        return SOFTMAX_ERR_CUDA;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
        *ok = true;
    } else if (a.type == cudaMemoryTypeHost) {
        *ok = a.devicePointer == p;
    } else {  // pageable host memory
        int dev = 0, pageable = 0, host_tables = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&host_tables, cudaDevAttrPageableMemoryAccessUsesHostPageTables, dev) !=
                cudaSuccess)
            return SOFTMAX_ERR_CUDA;
        *ok = pageable != 0 && host_tables != 0;
    }
    return SOFTMAX_OK;
}

}  // namespace

extern "C" {

int softmax_fwd(const void *in, void *out, int64_t rows, int64_t cols, int64_t row_stride, int dtype,
                cudaStream_t stream) {
    int64_t ext = 0;
    const uint64_t ia = (uint64_t)(uintptr_t)in, oa = (uint64_t)(uintptr_t)out;
    int st = check_args(ia, oa, rows, cols, row_stride, dtype, &ext);
    if (st != SOFTMAX_OK || rows == 0) return st;
    int sms = 0;
    st = device_sms(&sms);
    if (st != SOFTMAX_OK) return st;
    Plan p;
    st = plan_call(ia, oa, rows, cols, row_stride, dtype, sms, &p, nullptr);
    if (st != SOFTMAX_OK) return st;
    LaunchArgs a{in, out, rows, cols, row_stride, dtype, p.vec_store, stream, g_overlap.load(), p.whole};
    st = run(p, a);
    if (st == SOFTMAX_ERR_UNSUPPORTED && p.path == SOFTMAX_PATH_GRID && forced_shape().path != SOFTMAX_PATH_GRID) {
        // the grid path's counter cannot live in this `out` (host memory
        // without native atomics): the streaming cluster instead
        st = make_plan(ia, oa, rows, cols, row_stride, dtype, sms, Shape{SOFTMAX_PATH_STREAM, 0, 0, 0}, &p);
        if (st != SOFTMAX_OK) return st;
        st = run(p, a);
    }
    if (st == SOFTMAX_OK) g_last_path.store(p.path);
    return st;
}

int softmax_fwd_masked(const void *in, void *out, int64_t rows, int64_t cols, int64_t row_stride, int dtype,
                       float scale, int64_t causal_offset, int64_t rows_per_seq, cudaStream_t stream) {
    int64_t ext = 0;
    const uint64_t ia = (uint64_t)(uintptr_t)in, oa = (uint64_t)(uintptr_t)out;
    int st = check_args(ia, oa, rows, cols, row_stride, dtype, &ext);
    if (st != SOFTMAX_OK || rows == 0) return st;
    if (!(scale > 0.f) || !std::isfinite(scale) || rows_per_seq < 0) return SOFTMAX_ERR_ARG;
    int sms = 0;
    st = device_sms(&sms);
    if (st != SOFTMAX_OK) return st;
    Shape want = forced_shape();
    if (want.path != SOFTMAX_PATH_AUTO && want.path != SOFTMAX_PATH_WARP && want.path != SOFTMAX_PATH_CTA &&
        want.path != SOFTMAX_PATH_STREAM)
        want = Shape{SOFTMAX_PATH_STREAM, 0, 0, 0};  // no masked variant: the streaming cluster
    Plan p;
    st = make_plan(ia, oa, rows, cols, row_stride, dtype, sms, want, &p);
    if (st != SOFTMAX_OK) return st;
    if (p.path != SOFTMAX_PATH_WARP && p.path != SOFTMAX_PATH_CTA && p.path != SOFTMAX_PATH_STREAM) {
        // rows too long for a block: the streaming cluster, at its own shape
        st = make_plan(ia, oa, rows, cols, row_stride, dtype, sms, Shape{SOFTMAX_PATH_STREAM, 0, 0, 0}, &p);
        if (st != SOFTMAX_OK) return st;
    }
    LaunchArgs a{in, out, rows, cols, row_stride, dtype, p.vec_store, stream, g_overlap.load(), p.whole};
    // bounds that keep (r mod rows_per_seq) + off + 1 clear of int64 overflow
    const int64_t lim = (int64_t)1 << 62;
    a.mask.off = std::max(-lim, std::min(causal_offset, cols));
    a.mask.period = rows_per_seq;
    a.mask.k = (float)((double)scale * 1.4426950408889634);  // scale * log2 e, rounded once
    cudaError_t e = cudaSuccess;
    switch (p.path) {
        case SOFTMAX_PATH_WARP: e = launch_warp_masked(a, p.threads, p.group, p.vpt, p.grid); break;
        case SOFTMAX_PATH_CTA: e = launch_cta_masked(a, p.threads, p.vpt, p.grid); break;
        default: e = launch_stream_masked(a, p.threads, p.vpt, p.group, g_wait_ns.load(), g_starve.load()); break;
    }
    if (e == cudaErrorInvalidValue) return SOFTMAX_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return SOFTMAX_ERR_CUDA;
    g_last_path.store(p.path);
    return SOFTMAX_OK;
}

int softmax_masked_copy(const void *in, void *out, int64_t rows, int64_t cols, int64_t row_stride, int dtype,
                        int64_t causal_offset, int64_t rows_per_seq, int threads, cudaStream_t stream) {
    int64_t ext = 0;
    const uint64_t ia = (uint64_t)(uintptr_t)in, oa = (uint64_t)(uintptr_t)out;
    int st = check_args(ia, oa, rows, cols, row_stride, dtype, &ext);
    if (st != SOFTMAX_OK || rows == 0) return st;
    if (rows_per_seq < 0) return SOFTMAX_ERR_ARG;
    if (threads == 0) threads = 256;
    if (threads < 32 || threads > 1024 || (threads & (threads - 1)) != 0) return SOFTMAX_ERR_ARG;
    const int es = elem_bytes(dtype);
    if (ia % kVecBytes != 0 || oa % kVecBytes != 0 || (row_stride * es) % kVecBytes != 0 ||
        (cols * es) % kVecBytes != 0)
        return SOFTMAX_ERR_UNSUPPORTED;  // rows of whole 16-byte vectors only
    LaunchArgs a{in, out, rows, cols, row_stride, dtype, 1, stream, g_overlap.load(), 1};
    const int64_t lim = (int64_t)1 << 62;
    a.mask.off = std::max(-lim, std::min(causal_offset, cols));
    a.mask.period = rows_per_seq;
    const cudaError_t e = launch_masked_copy(a, threads, std::min<int64_t>(rows, kMaxGrid));
    if (e == cudaErrorInvalidValue) return SOFTMAX_ERR_UNSUPPORTED;
    return e == cudaSuccess ? SOFTMAX_OK : SOFTMAX_ERR_CUDA;
}

int64_t softmax_host_workspace_bytes(int64_t rows, int64_t cols, int64_t row_stride, int dtype,
                                     int64_t chunk_bytes) {
    if (dtype != SOFTMAX_F32 && dtype != SOFTMAX_F16 && dtype != SOFTMAX_BF16) return -SOFTMAX_ERR_DTYPE;
    if (rows < 0 || cols < 1) return -SOFTMAX_ERR_SHAPE;
    if (row_stride < cols) return -SOFTMAX_ERR_STRIDE;
    if (rows == 0) return 0;
    const int es = elem_bytes(dtype);
    if (row_stride > INT64_MAX / 4 / es) return -SOFTMAX_ERR_SHAPE;
    const int64_t quarter = rows * cols * es / 4;
    const int64_t def = std::min(kHostChunkMax, std::max(kHostChunkMin, quarter));
    const int64_t cr = host_chunk_rows(rows, cols, es, chunk_bytes > 0 ? chunk_bytes : def);
    return kHostSlots * host_slot_bytes(cr, cols, es);
}

int softmax_fwd_host(const void *in_host, void *out_host, int64_t rows, int64_t cols, int64_t row_stride,
                     int dtype, void *workspace, int64_t workspace_bytes, cudaStream_t stream) {
    int64_t ext = 0;
    const uint64_t ia = (uint64_t)(uintptr_t)in_host, oa = (uint64_t)(uintptr_t)out_host;
    int st = check_args(ia, oa, rows, cols, row_stride, dtype, &ext);
    if (st != SOFTMAX_OK || rows == 0) return st;
    if (!workspace && workspace_bytes == 0) {
        // zero-copy: the kernels read and write the host buffers in place,
        // the bytes crossing the CPU-GPU link inside them
        // (the first and the last byte of each range: one allocation may end
        // before the range does)
        const char *ends[4] = {static_cast<const char *>(in_host), static_cast<const char *>(in_host) + ext - 1,
                               static_cast<const char *>(out_host), static_cast<const char *>(out_host) + ext - 1};
        for (const char *e : ends) {
            bool ok = false;
            st = device_reaches(e, &ok);
            if (st != SOFTMAX_OK) return st;
            if (!ok) return SOFTMAX_ERR_ARG;
        }
        return softmax_fwd(in_host, out_host, rows, cols, row_stride, dtype, stream);
    }
    if (!workspace) return SOFTMAX_ERR_NULL;
    if ((uintptr_t)workspace % 256 != 0 || workspace_bytes < 0) return SOFTMAX_ERR_ARG;
    const int es = elem_bytes(dtype);
    // the largest chunk (up to the default) of which three fit the workspace
    // chunks as large as the workspace's three slots allow (its size sets the
    // pipeline's granularity: softmax_host_workspace_bytes)
    const int64_t fit = workspace_bytes / kHostSlots / 256 * 256 / es;  // elements per slot
    if (fit < cols) return SOFTMAX_ERR_ARG;
    const int64_t cr = std::min(rows, fit / cols);
    const int64_t sb = host_slot_bytes(cr, cols, es);
    int sms = 0, dev = 0;
    st = device_sms(&sms);
    if (st != SOFTMAX_OK) return st;
    if (cudaGetDevice(&dev) != cudaSuccess) return SOFTMAX_ERR_CUDA;

    HostPipe &hp = g_host_pipes[dev & (kMaxDevices - 1)];
    std::lock_guard<std::mutex> lock(hp.mu);
    if (host_pipe_ready(hp) != cudaSuccess) return SOFTMAX_ERR_CUDA;
    cudaError_t e = cudaEventRecord(hp.start, stream);
    for (int j = 0; j < kHostSlots && e == cudaSuccess; ++j) e = cudaStreamWaitEvent(hp.s[j], hp.start, 0);
    if (e != cudaSuccess) return SOFTMAX_ERR_CUDA;
    const size_t row_bytes = (size_t)(row_stride * es), data_bytes = (size_t)(cols * es);
    int path = 0;
    for (int64_t r0 = 0, i = 0; r0 < rows && st == SOFTMAX_OK; r0 += cr, ++i) {
        const int j = (int)(i % kHostSlots);
        const int64_t n = std::min(cr, rows - r0);
        char *slot = static_cast<char *>(workspace) + j * sb;
        // the rows' data only: pitched copies skip the host rows' padding
        const char *src = static_cast<const char *>(in_host) + r0 * row_bytes;
        const cudaError_t ce = row_bytes == data_bytes
                                   ? cudaMemcpyAsync(slot, src, data_bytes * n, cudaMemcpyHostToDevice, hp.s[j])
                                   : cudaMemcpy2DAsync(slot, data_bytes, src, row_bytes, data_bytes, (size_t)n,
                                                       cudaMemcpyHostToDevice, hp.s[j]);
        if (ce != cudaSuccess) {
            st = SOFTMAX_ERR_CUDA;
            break;
        }
        const uint64_t sa = (uint64_t)(uintptr_t)slot;
        Plan p;
        st = plan_call(sa, sa, n, cols, cols, dtype, sms, &p, nullptr);
        if (st != SOFTMAX_OK) break;
        LaunchArgs a{slot, slot, n, cols, cols, dtype, p.vec_store, hp.s[j], g_overlap.load(), p.whole};
        st = run(p, a);  // in place in the slot
        if (st != SOFTMAX_OK) break;
        path = p.path;
        char *dst = static_cast<char *>(out_host) + r0 * row_bytes;
        const cudaError_t de = row_bytes == data_bytes
                                   ? cudaMemcpyAsync(dst, slot, data_bytes * n, cudaMemcpyDeviceToHost, hp.s[j])
                                   : cudaMemcpy2DAsync(dst, row_bytes, slot, data_bytes, data_bytes, (size_t)n,
                                                       cudaMemcpyDeviceToHost, hp.s[j]);
        if (de != cudaSuccess) st = SOFTMAX_ERR_CUDA;
    }
    // the caller's stream waits for all three slot streams, whatever happened
    for (int j = 0; j < kHostSlots; ++j) {
        if (cudaEventRecord(hp.done[j], hp.s[j]) != cudaSuccess ||
            cudaStreamWaitEvent(stream, hp.done[j], 0) != cudaSuccess)
            st = SOFTMAX_ERR_CUDA;
    }
    if (st == SOFTMAX_OK) g_last_path.store(path);
    return st;
}

int softmax_fwd_noalloc(const void *in, void *out, int64_t rows, int64_t cols, int64_t row_stride, int dtype,
                        cudaStream_t stream) {
    int64_t ext = 0;
    const uint64_t ia = (uint64_t)(uintptr_t)in, oa = (uint64_t)(uintptr_t)out;
    int st = check_args(ia, oa, rows, cols, row_stride, dtype, &ext);
    if (st != SOFTMAX_OK || rows == 0) return st;
    int sms = 0;
    st = device_sms(&sms);
    if (st != SOFTMAX_OK) return st;
    int64_t chunks = 0, chunk_vecs = 0, grid = 0;
    st = plan_noalloc(ia, rows, cols, row_stride, dtype, sms, &chunks, &chunk_vecs, &grid);
    if (st != SOFTMAX_OK) return st;
    const int vec_store = (ia % kVecBytes) == (oa % kVecBytes);
    LaunchArgs a{in, out, rows, cols, row_stride, dtype, vec_store, stream, g_overlap.load(), 0};
    const cudaError_t e = launch_split_noalloc(a, chunks, chunk_vecs, grid);
    if (e == cudaErrorInvalidValue) return SOFTMAX_ERR_SCRATCH_LIMIT;
    return e == cudaSuccess ? SOFTMAX_OK : SOFTMAX_ERR_CUDA;
}

const char *softmax_status_string(int status) {
    switch (status) {
        case SOFTMAX_OK: return "ok";
        case SOFTMAX_ERR_NULL: return "null pointer with rows > 0";
        case SOFTMAX_ERR_SHAPE: return "bad shape (rows < 0, cols < 1, or extent overflows int64)";
        case SOFTMAX_ERR_STRIDE: return "row_stride < cols";
        case SOFTMAX_ERR_DTYPE: return "unknown dtype";
        case SOFTMAX_ERR_OVERLAP: return "in and out overlap without being equal";
        case SOFTMAX_ERR_UNSUPPORTED: return "forced path or shape cannot take these arguments";
        case SOFTMAX_ERR_CUDA: return "CUDA runtime error";
        case SOFTMAX_ERR_TIMEOUT: return "a bounded device wait ran out";
        case SOFTMAX_ERR_ALIGN: return "pointer not aligned to its element size";
        case SOFTMAX_ERR_ARG: return "bad argument to a diagnostic call";
        case SOFTMAX_ERR_SCRATCH_LIMIT:
            return "softmax_fwd_noalloc: more rows than its fixed device scratch array holds states for";
        default: return "unknown status";
    }
}

int softmax_last_path(void) { return g_last_path.load(); }

int softmax_set_force_path(int path, int threads, int vpt, int group) {
    if (path < SOFTMAX_PATH_AUTO || path > SOFTMAX_PATH_GRID || path == SOFTMAX_PATH_SPLIT || path == 5)
        return SOFTMAX_ERR_ARG;
    g_force_path.store(path);
    g_force_threads.store(threads > 0 ? threads : 0);
    g_force_vpt.store(vpt > 0 ? vpt : 0);
    g_force_group.store(group > 0 ? group : 0);
    return SOFTMAX_OK;
}

int softmax_plan(uint64_t in_addr, uint64_t out_addr, int64_t rows, int64_t cols, int64_t row_stride, int dtype,
                 int num_sms, softmax_plan_t *plan) {
    if (!plan || num_sms < 0) return SOFTMAX_ERR_ARG;
    std::memset(plan, 0, sizeof(*plan));
    int64_t ext = 0;
    int st = check_args(in_addr, out_addr, rows, cols, row_stride, dtype, &ext);
    if (st != SOFTMAX_OK || rows == 0) return st;
    int sms = num_sms;
    if (sms == 0) {
        st = device_sms(&sms);
        if (st != SOFTMAX_OK) return st;
    }
    Plan p;
    st = plan_call(in_addr, out_addr, rows, cols, row_stride, dtype, sms, &p, nullptr);
    if (st != SOFTMAX_OK) return st;
    fill_public_plan(p, plan);
    return SOFTMAX_OK;
}

int softmax_check_device_error(cudaStream_t stream) {
    unsigned int word = 0;
    if (read_clear_error_word(stream, &word) != cudaSuccess) return SOFTMAX_ERR_CUDA;
    unsigned int attn_word = 0;
    if (attn::read_clear_attn_error_word(&attn_word) != cudaSuccess) return SOFTMAX_ERR_CUDA;
    if (word & kErrNotCluster) return SOFTMAX_ERR_CUDA;
    return (word | attn_word) ? SOFTMAX_ERR_TIMEOUT : SOFTMAX_OK;
}

int softmax_set_wait_test(int64_t wait_limit_ns, int starve) {
    // a drain wait lasts twice the limit and must stay under 2^31 ns
    g_wait_ns.store(wait_limit_ns > 0 ? std::min(wait_limit_ns, kDefaultWaitNs) : kDefaultWaitNs);
    g_starve.store(starve ? 1 : 0);
    return SOFTMAX_OK;
}

int softmax_set_launch_overlap(int enable) {
    g_overlap.store(enable ? 1 : 0);
    return SOFTMAX_OK;
}

int softmax_tune_candidates(uint64_t in_addr, uint64_t out_addr, int64_t rows, int64_t cols, int64_t row_stride,
                            int dtype, int num_sms, softmax_shape_t *shapes, int capacity) {
    (void)num_sms;  // the candidate set depends on the row geometry only
    if (capacity < 0 || (capacity > 0 && !shapes)) return -SOFTMAX_ERR_ARG;
    int64_t ext = 0;
    const int st = check_args(in_addr, out_addr, rows, cols, row_stride, dtype, &ext);
    if (st != SOFTMAX_OK) return -st;
    const std::vector<Shape> c = candidates_for(in_addr, out_addr, cols, row_stride, dtype);
    for (int i = 0; i < (int)c.size() && i < capacity; ++i)
        shapes[i] = softmax_shape_t{c[i].path, c[i].threads, c[i].vpt, c[i].group};
    return (int)c.size();
}

int softmax_autotune(const void *in, void *out, int64_t rows, int64_t cols, int64_t row_stride, int dtype,
                     cudaStream_t stream, int iters, softmax_tune_result_t *result) {
    if (result) std::memset(result, 0, sizeof(*result));
    int64_t ext = 0;
    const uint64_t ia = (uint64_t)(uintptr_t)in, oa = (uint64_t)(uintptr_t)out;
    int st = check_args(ia, oa, rows, cols, row_stride, dtype, &ext);
    if (st != SOFTMAX_OK || rows == 0) return st;
    if (ia == oa) return SOFTMAX_ERR_ARG;  // every candidate must see the same input
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return SOFTMAX_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return SOFTMAX_ERR_ARG;
    if (iters <= 0) iters = 20;
    int sms = 0, dev = 0;
    st = device_sms(&sms);
    if (st != SOFTMAX_OK) return st;
    if (cudaGetDevice(&dev) != cudaSuccess) return SOFTMAX_ERR_CUDA;

    cudaEvent_t ev[2] = {nullptr, nullptr};
    if (cudaEventCreate(&ev[0]) != cudaSuccess || cudaEventCreate(&ev[1]) != cudaSuccess) {
        if (ev[0]) cudaEventDestroy(ev[0]);
        return SOFTMAX_ERR_CUDA;
    }
    const std::vector<Shape> cands = candidates_for(ia, oa, cols, row_stride, dtype);
    Plan best_plan;
    double best_us = 0.0, auto_us = 0.0;
    int timed = 0;
    bool have = false, best_is_auto = false;
    st = SOFTMAX_OK;
    for (size_t i = 0; i < cands.size() && st == SOFTMAX_OK; ++i) {
        Plan p;
        if (make_plan(ia, oa, rows, cols, row_stride, dtype, sms, cands[i], &p) != SOFTMAX_OK) continue;
        LaunchArgs a{in, out, rows, cols, row_stride, dtype, p.vec_store, stream, g_overlap.load(), p.whole};
        if (run(p, a) != SOFTMAX_OK || run(p, a) != SOFTMAX_OK) continue;  // a shape the launchers refuse
        if (cudaEventRecord(ev[0], stream) != cudaSuccess) {
            st = SOFTMAX_ERR_CUDA;
            break;
        }
        for (int k = 0; k < iters && st == SOFTMAX_OK; ++k) st = run(p, a);
        float ms = 0.f;
        if (st != SOFTMAX_OK || cudaEventRecord(ev[1], stream) != cudaSuccess ||
            cudaEventSynchronize(ev[1]) != cudaSuccess || cudaEventElapsedTime(&ms, ev[0], ev[1]) != cudaSuccess) {
            st = SOFTMAX_ERR_CUDA;
            break;
        }
        const double us = 1000.0 * ms / iters;
        ++timed;
        if (i == 0) auto_us = us;
        // another shape replaces the automatic one only when it is at least 2%
        // faster (run-to-run noise of these timings is about 1%)
        if (!have || us < (best_is_auto ? 0.98 * best_us : best_us)) {
            best_is_auto = i == 0;
            have = true;
            best_us = us;
            best_plan = p;
        }
    }
    cudaEventDestroy(ev[0]);
    cudaEventDestroy(ev[1]);
    if (st != SOFTMAX_OK) return st;
    if (!have) return SOFTMAX_ERR_UNSUPPORTED;
    store_tuned(tune_key(dev, ia, oa, rows, cols, row_stride, dtype),
                Shape{best_plan.path, best_plan.threads, best_plan.vpt, best_plan.group});
    if (result) {
        fill_public_plan(best_plan, &result->plan);
        result->best_us = best_us;
        result->auto_us = auto_us;
        result->candidates = timed;
    }
    return SOFTMAX_OK;
}

int softmax_autotune_size(void) {
    std::lock_guard<std::mutex> lock(g_tune_mu);
    return (int)g_tuned.size();
}

int softmax_autotune_clear(void) {
    std::lock_guard<std::mutex> lock(g_tune_mu);
    g_tuned.clear();
    g_tuned_count.store(0);
    return SOFTMAX_OK;
}

int softmax_abi_version(void) { return kAbiVersion; }

}  // extern "C"

namespace mbrs {
int host_device_sms(int *sms) { return device_sms(sms); }
int64_t host_wait_ns() { return g_wait_ns.load(); }
}  // namespace mbrs
