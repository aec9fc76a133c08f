// kernels.cuh -- the four row-softmax kernels (templates; instantiated per path
// in k_*.cu).
//
//   path 1  k_warp_rows     G lanes (2..32) own a row, VPT vectors per lane;
//                           shuffle-only reduction, no shared memory.
//   path 2  k_cta_rows      a block owns a row held in registers; warp
//                           shuffles, then one shared-memory exchange.
//   path 3  k_cluster_rows  a cluster of blocks owns a row; each block pulls
//                           its slice with a TMA bulk copy, and the blocks
//                           exchange their (max, sum) through distributed
//                           shared memory -- still one read, one write.
//   path 4  k_split_stats / k_split_apply
//                           rows cut into chunks spread over the whole grid;
//                           pass 1 streams each chunk into a (max, sum) state
//                           in scratch, pass 2 merges a row's states, re-reads
//                           its chunk and writes it (the two-pass form that a
//                           reduction spanning many blocks needs: page
//                           "Kernel Fusion", section "What fusion cannot fix").
//
// All paths keep the per-thread (s_t, l_t) scheme of common.cuh: one exp per
// element, one merge round per row.  Variables named m / M below hold the
// base-2 shifts s / S of those states.
#pragma once

#include "common.cuh"

namespace mbrs {

// ---------------------------------------------------------------------------
// path 1: a lane group per row
// ---------------------------------------------------------------------------
template <typename T, int G, int VPT>
__global__ void __launch_bounds__(256) k_warp_rows(const T *in, T *out, int64_t rows, int64_t cols,
                                                   int64_t stride, int vec_store) {
    static_assert(G >= 2 && G <= 32 && (G & (G - 1)) == 0, "lane group is a power of two");
    const int t = threadIdx.x & (G - 1);
    const int64_t groups_per_block = blockDim.x / G;
    const int64_t row_step = (int64_t)gridDim.x * groups_per_block;
    // rows of this warp's first group; the loop bound is warp-uniform so that
    // every lane reaches every shuffle
    const int64_t warp_row0 = (int64_t)blockIdx.x * groups_per_block + (threadIdx.x & ~31) / G;
    for (int64_t base = warp_row0; base < rows; base += row_step) {
        const int64_t row = base + (threadIdx.x & 31) / G;
        const bool active = row < rows;
        RowView<T> rv(in + (active ? row : 0) * stride, out + (active ? row : 0) * stride, cols,
                      vec_store != 0);
        Tile<T, VPT> tile;
        tile.load(rv, t, G, active ? rv.nvec : 0);
        const float2 s = tile.exp_in_place();
        float m = s.x, l = s.y;
        group_merge<G>(m, l);
        if (active) tile.scale_store(rv, t, G, rv.nvec, out_factor(s.x, m, l));
    }
}

// ---------------------------------------------------------------------------
// path 2: a block per row
// ---------------------------------------------------------------------------
template <int NW>
__device__ __forceinline__ void block_merge(float &m, float &l, float2 *red) {
    // red: NW slots; caller double-buffers across rows
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    group_merge<32>(m, l);
    if (lane == 0) red[warp] = make_float2(m, l);
    __syncthreads();
    const float2 w = lane < NW ? red[lane] : make_float2(-INFINITY, 0.f);
    m = w.x;
    l = w.y;
    group_merge<32>(m, l);
}

template <typename T, int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS) k_cta_rows(const T *in, T *out, int64_t rows, int64_t cols,
                                                      int64_t stride, int vec_store) {
    constexpr int NW = THREADS / 32;
    __shared__ float2 red[2][NW];
    int parity = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, parity ^= 1) {
        RowView<T> rv(in + row * stride, out + row * stride, cols, vec_store != 0);
        Tile<T, VPT> tile;
        tile.load(rv, threadIdx.x, THREADS, rv.nvec);
        const float2 s = tile.exp_in_place();
        float m = s.x, l = s.y;
        block_merge<NW>(m, l, red[parity]);
        tile.scale_store(rv, threadIdx.x, THREADS, rv.nvec, out_factor(s.x, m, l));
    }
}

// ---------------------------------------------------------------------------
// path 3: a cluster per row
// ---------------------------------------------------------------------------
constexpr int kMaxCluster = 16;
constexpr uint32_t kBulkPiece = 16384;  // bytes per cp.async.bulk

// The device error word that bounded waits set when they run out.  Each
// translation unit has its own copy; the cluster path's unit (the only one
// with waits) owns the reader.
static __device__ unsigned int g_error_word = 0;

template <int THREADS, int VPT>
struct ClusterSmem {
    static constexpr int kStageBytes = THREADS * VPT * kVecBytes;
    static constexpr int kBarOff = kStageBytes;
    static constexpr int kRedOff = kBarOff + 16;
    static constexpr int kSlotOff = kRedOff + (THREADS / 32) * 8;
    static constexpr int kBytes = kSlotOff + kMaxCluster * 8;
};

template <typename T, int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS, (THREADS >= 1024 ? 1 : 1024 / THREADS))
    k_cluster_rows(const T *in, T *out, int64_t rows, int64_t cols, int64_t stride, int vec_store,
                   int64_t wait_ns, int starve) {
    constexpr int V = Elem<T>::kVec;
    constexpr int NW = THREADS / 32;
    using L = ClusterSmem<THREADS, VPT>;
    extern __shared__ __align__(128) unsigned char smem[];
    const uint4 *stage = reinterpret_cast<const uint4 *>(smem);
    float2 *red = reinterpret_cast<float2 *>(smem + L::kRedOff);
    float2 *slots = reinterpret_cast<float2 *>(smem + L::kSlotOff);
    const uint32_t bar = smem_addr(smem + L::kBarOff);
    const int tid = threadIdx.x, lane = tid & 31;

    const uint32_t rank = cluster_rank(), csize = cluster_size();
    const int64_t row = blockIdx.x / csize;
    RowView<T> rv(in + row * stride, out + row * stride, cols, vec_store != 0);

    // this block's slice of the row's vectors, and the part of it made of whole
    // vectors (the only part a bulk copy may move: 16-byte aligned, inside the row)
    const int64_t per = (rv.nvec + csize - 1) / csize;
    const int64_t s0 = min((int64_t)rank * per, rv.nvec), s1 = min(s0 + per, rv.nvec);
    const int64_t first_full = rv.head > 0 ? 1 : 0;
    const int64_t full_end = ((rv.head + cols) % V) != 0 ? rv.nvec - 1 : rv.nvec;
    const int64_t f0 = max(s0, first_full), f1 = min(s1, full_end);
    const uint32_t bytes = f1 > f0 ? (uint32_t)((f1 - f0) * kVecBytes) : 0u;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0 && !starve) {
        if (bytes > 0) {
            mbar_arrive_expect_tx(bar, bytes);
            const char *src = reinterpret_cast<const char *>(rv.in + (f0 * V - rv.head));
            const uint32_t dst = smem_addr(stage + (f0 - s0));
            for (uint32_t off = 0; off < bytes; off += kBulkPiece)
                bulk_g2s(dst + off, src + off, min(kBulkPiece, bytes - off), bar);
        } else {
            mbar_arrive(bar);
        }
    }
    // announce that this block runs: peers may write into its shared memory
    // once they have waited on this arrival
    __syncwarp();
    cluster_arrive_relaxed();

    bool ok = mbar_wait_bounded(bar, 0, wait_ns);
    if (!ok) {
        atomicOr(&g_error_word, kErrWaitTimeout);
        // a copy may still be landing in this block's shared memory: give it
        // one more bounded wait before the memory is reused or released
        if (!starve) mbar_wait_bounded(bar, 0, wait_ns);
    }

    Tile<T, VPT> tile;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t v = s0 + j * THREADS + tid;
        if (v < s1) {
            if (v >= f0 && v < f1)
                Elem<T>::unpack(stage[v - s0], tile.x[j]);
            else
                rv.load(v, tile.x[j]);  // a partial vector at the row's edge
        } else {
#pragma unroll
            for (int i = 0; i < V; ++i) tile.x[j][i] = -INFINITY;
        }
    }
    const float2 s = tile.exp_in_place();
    float m = s.x, l = s.y;
    block_merge<NW>(m, l, red);

    // push this block's state into every block of the cluster, then gather
    cluster_wait_acquire();
    if (tid == 0) {
        const uint32_t my_slot = smem_addr(slots + rank);
        for (uint32_t q = 0; q < csize; ++q) st_cluster_f2(map_to_rank(my_slot, q), m, l);
    }
    __syncwarp();
    cluster_arrive_release();
    cluster_wait_acquire();
    const float2 w = lane < (int)csize ? slots[lane] : make_float2(-INFINITY, 0.f);
    m = w.x;
    l = w.y;
    group_merge<32>(m, l);
    if (ok) tile.scale_store(rv, s0 + tid, THREADS, s1, out_factor(s.x, m, l));
}

// ---------------------------------------------------------------------------
// path 4: rows split over the grid (two passes, states in scratch)
// ---------------------------------------------------------------------------
template <typename T, int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS) k_split_stats(const T *in, int64_t rows, int64_t cols, int64_t stride,
                                                         int64_t chunks, int64_t chunk_vecs, float2 *part) {
    constexpr int NW = THREADS / 32;
    constexpr int64_t kTile = (int64_t)THREADS * VPT;
    __shared__ float2 red[2][NW];
    int parity = 0;
    const int64_t units = rows * chunks;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x, parity ^= 1) {
        const int64_t row = u / chunks, k = u - row * chunks;
        RowView<T> rv(in + row * stride, nullptr, cols, false);
        const int64_t c0 = min(k * chunk_vecs, rv.nvec), c1 = min(c0 + chunk_vecs, rv.nvec);
        float m = -INFINITY, l = 0.f;
        for (int64_t t0 = c0; t0 < c1; t0 += kTile) {
            Tile<T, VPT> tile;
            tile.load(rv, t0 + threadIdx.x, THREADS, c1);
            const float2 s = tile.exp_in_place();
            const float M = fmaxf(m, s.x);
            l = rescale(l, m, M) + rescale(s.y, s.x, M);
            m = M;
        }
        block_merge<NW>(m, l, red[parity]);
        if (threadIdx.x == 0) part[u] = make_float2(m, l);
    }
}

template <typename T, int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS)
    k_split_apply(const T *in, T *out, int64_t rows, int64_t cols, int64_t stride, int64_t chunks,
                  int64_t chunk_vecs, const float2 *part, int vec_store) {
    constexpr int V = Elem<T>::kVec;
    constexpr int NW = THREADS / 32;
    constexpr int64_t kTile = (int64_t)THREADS * VPT;
    __shared__ float2 red[2][NW];
    int parity = 0;
    const int64_t units = rows * chunks;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x, parity ^= 1) {
        const int64_t row = u / chunks, k = u - row * chunks;
        RowView<T> rv(in + row * stride, out + row * stride, cols, vec_store != 0);
        const int64_t c0 = min(k * chunk_vecs, rv.nvec), c1 = min(c0 + chunk_vecs, rv.nvec);
        Tile<T, VPT> tile;
        tile.load(rv, c0 + threadIdx.x, THREADS, c1);  // in flight while the states merge
        float m = -INFINITY, l = 0.f;
        for (int64_t i = threadIdx.x; i < chunks; i += THREADS) {
            const float2 p = part[row * chunks + i];
            const float M = fmaxf(m, p.x);
            l = rescale(l, m, M) + rescale(p.y, p.x, M);
            m = M;
        }
        block_merge<NW>(m, l, red[parity]);
        const float shift = m;  // states are (s, l): m here is the row's S
        const float inv = m == -INFINITY ? __int_as_float(0x7fc00000) : 1.f / l;
        for (int64_t t0 = c0; t0 < c1; t0 += kTile) {
            if (t0 != c0) tile.load(rv, t0 + threadIdx.x, THREADS, c1);
#pragma unroll
            for (int j = 0; j < VPT; ++j)
#pragma unroll
                for (int i = 0; i < V; ++i) tile.x[j][i] = ex2(fmaf(tile.x[j][i], kLog2e, -shift)) * inv;
            tile.scale_store(rv, t0 + threadIdx.x, THREADS, c1, 1.f);
        }
    }
}

}  // namespace mbrs
