// kernels.cuh -- the row-softmax kernels (templates; instantiated per path
// in k_*.cu).
//
//   path 1  k_warp_rows     G lanes (2..32) own a row, VPT vectors per lane;
//                           shuffle-only reduction, no shared memory.
//   path 2  k_cta_rows      a block owns a row held in registers; warp
//                           shuffles, then one shared-memory exchange.
//   path 3  k_cluster_rows  a cluster of blocks owns a row, each block holding
//                           its slice in registers; the blocks exchange their
//                           (max, sum) through distributed shared memory --
//                           still one read, one write.
//   path 6  k_cluster_stream
//                           a cluster of blocks owns a row of any length and
//                           streams its slices twice (states exchanged in
//                           distributed shared memory between the passes).
//   path 7  k_packed_rows   narrow dense rows staged through shared memory,
//                           one thread per row.
//   path 8  k_grid_stats / k_grid_apply
//                           a few very long rows cut into chunks over the
//                           whole grid (out != in): the chunk states go into
//                           the start of the output row, and the second
//                           launch folds them, counts its blocks on an atomic
//                           counter there and writes (two passes and an
//                           atomic: page "Kernel Fusion", section "What
//                           fusion cannot fix").
//   k_split_stats / k_split_apply
//                           rows cut into chunks spread over the whole grid;
//                           pass 1 streams each chunk into a (max, sum) state
//                           in a global array, pass 2 merges a row's states,
//                           re-reads its chunk and writes it (the two-pass
//                           form that a reduction spanning many blocks needs:
//                           page "Kernel Fusion", section "What fusion cannot
//                           fix").  Only softmax_fwd_noalloc runs them, with
//                           the states in a fixed array inside the library.
//
// All paths keep the per-thread (s_t, l_t) scheme of common.cuh: one exp per
// element, one merge round per row.  Variables named m / M below hold the
// base-2 shifts s / S of those states.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace mbrs {

// ---------------------------------------------------------------------------
// path 1: a lane group per row
// ---------------------------------------------------------------------------
template <typename T, int G, int VPT, bool WHOLE>
__global__ void __launch_bounds__(256) k_warp_rows(const T *in, T *out, int64_t rows, int64_t cols,
                                                   int64_t stride, int vec_store) {
    static_assert(G >= 2 && G <= 32 && (G & (G - 1)) == 0, "lane group is a power of two");
    const int t = threadIdx.x & (G - 1);
    const int64_t groups_per_block = blockDim.x / G;
    const int64_t row_step = (int64_t)gridDim.x * groups_per_block;
    // rows of this warp's first group; the loop bound is warp-uniform so that
    // every lane reaches every shuffle
    const int64_t warp_row0 = (int64_t)blockIdx.x * groups_per_block + (threadIdx.x & ~31) / G;
    if (t == 0 && warp_row0 + (threadIdx.x & 31) / G < rows)
        prefetch_span_l2(in + (warp_row0 + (threadIdx.x & 31) / G) * stride, 0, cols, cols);
    pdl_enter();
    for (int64_t base = warp_row0; base < rows; base += row_step) {
        const int64_t row = base + (threadIdx.x & 31) / G;
        const bool active = row < rows;
        RowView<T> rv(in + (active ? row : 0) * stride, out + (active ? row : 0) * stride, cols,
                      vec_store != 0);
        Tile<T, VPT> tile;
        tile.template load<WHOLE>(rv, t, G, active ? rv.nvec : 0);
        const float2 s = tile.stats();
        float m = s.x, l = s.y;
        group_merge<G>(m, l);
        if (active) tile.template scale_store<WHOLE>(rv, t, G, rv.nvec, out_factor(s.x, m, l));
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

template <typename T, int THREADS, int VPT, bool WHOLE>
__device__ __forceinline__ void cta_rows_body(const T *in, T *out, int64_t rows, int64_t cols, int64_t stride,
                                              int vec_store) {
    constexpr int NW = THREADS / 32;
    __shared__ float2 red[2][NW];
    if (threadIdx.x == 0 && blockIdx.x < rows) prefetch_span_l2(in + blockIdx.x * stride, 0, cols, cols);
    pdl_enter();
    int parity = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, parity ^= 1) {
        RowView<T> rv(in + row * stride, out + row * stride, cols, vec_store != 0);
        Tile<T, VPT> tile;
        tile.template load<WHOLE>(rv, threadIdx.x, THREADS, rv.nvec);
        const float2 s = tile.stats();
        float m = s.x, l = s.y;
        block_merge<NW>(m, l, red[parity]);
        tile.template scale_store<WHOLE>(rv, threadIdx.x, THREADS, rv.nvec, out_factor(s.x, m, l));
    }
}

// Up to 5 vectors per thread: the compiler's own register choice (an explicit
// minimum of one block per SM lets it take more: 64 instead of 40 registers
// for 64 threads x 4 fp16 vectors).
template <typename T, int THREADS, int VPT, bool WHOLE>
__global__ void __launch_bounds__(THREADS) k_cta_rows(const T *in, T *out, int64_t rows, int64_t cols,
                                                      int64_t stride, int vec_store) {
    cta_rows_body<T, THREADS, VPT, WHOLE>(in, out, rows, cols, stride, vec_store);
}

// 6 or more vectors per thread: bounded to 64 registers (1024 threads per SM),
// so that such wide rows still have two in flight per SM.
template <typename T, int THREADS, int VPT, bool WHOLE>
__global__ void __launch_bounds__(THREADS, 1024 / THREADS)
    k_cta_rows_wide(const T *in, T *out, int64_t rows, int64_t cols, int64_t stride, int vec_store) {
    cta_rows_body<T, THREADS, VPT, WHOLE>(in, out, rows, cols, stride, vec_store);
}

// ---------------------------------------------------------------------------
// path 3: a cluster per row
// ---------------------------------------------------------------------------
constexpr int kMaxCluster = 16;

// The device error word that bounded waits set when they run out.  Each
// translation unit has its own copy; the cluster paths' unit (the only one
// with waits) owns the reader.
static __device__ unsigned int g_error_word = 0;

// Shared memory of the cluster kernels: the state exchange barrier, the
// block-merge scratch and one exchange slot per cluster block.
template <int THREADS>
struct ClusterSmem {
    static constexpr int kXbarOff = 0;  // state exchange barrier
    static constexpr int kRedOff = 16;
    static constexpr int kSlotOff = kRedOff + (THREADS / 32) * 8;
    static constexpr int kBytes = kSlotOff + kMaxCluster * 8;
};

// Exchange a block's (s, l) state with every block of its cluster: st.async
// into slot `rank` of each peer (itself included), completing on the peer's
// exchange barrier `xbar` (armed for csize * 8 bytes), then a bounded wait for
// all csize states.  The caller has announced itself with a relaxed cluster
// arrive after initialising xbar; the cluster wait here makes sure every peer
// has done the same before any store targets it.  No block leaves before it
// has received every peer's state, so no store can reach a block that has
// gone.  Returns the merged row state in (m, l) on every thread; false when a
// wait ran out (then the block stays resident for as long as a late peer's
// waits can last).  starve != 0 (a test hook) sends nothing, so every wait of
// the cluster runs out and no store is in flight when the blocks leave.
template <int NW>
__device__ __forceinline__ bool cluster_exchange(float &m, float &l, float2 *slots, uint32_t xbar, uint32_t rank,
                                                 uint32_t csize, int64_t wait_ns, int starve) {
    const int lane = threadIdx.x & 31;
    cluster_wait_acquire();
    if (threadIdx.x == 0 && !starve) {
        const uint32_t my_slot = smem_addr(slots + rank);
        for (uint32_t q = 0; q < csize; ++q) st_async_f2(map_to_rank(my_slot, q), m, l, map_to_rank(xbar, q));
    }
    bool ok = true;
    if (!mbar_wait_bounded(xbar, 0, wait_ns)) {
        atomicOr(&g_error_word, kErrWaitTimeout);
        ok = false;
        mbar_wait_bounded(xbar, 0, 2 * wait_ns);
    }
    const float2 w = lane < (int)csize ? slots[lane] : make_float2(-INFINITY, 0.f);
    m = w.x;
    l = w.y;
    group_merge<32>(m, l);
    return ok;
}

// Each block loads its slice straight into registers (no staging, so
// occupancy is bounded by registers alone), reduces it, exchanges its state
// with the cluster and stores its slice.
template <typename T, int THREADS, int VPT, bool WHOLE>
__global__ void __launch_bounds__(THREADS, (THREADS >= 1024 ? 1 : 1024 / THREADS))
    k_cluster_rows(const T *in, T *out, int64_t rows, int64_t cols, int64_t stride, int vec_store,
                   int64_t wait_ns, int starve) {
    if (!explicit_cluster()) {  // launched without clusters: touch no cluster state
        pdl_enter();
        if (threadIdx.x == 0) atomicOr(&g_error_word, kErrNotCluster);
        return;
    }
    constexpr int V = Elem<T>::kVec;
    constexpr int NW = THREADS / 32;
    using L = ClusterSmem<THREADS>;
    extern __shared__ __align__(128) unsigned char smem[];
    float2 *red = reinterpret_cast<float2 *>(smem + L::kRedOff);
    float2 *slots = reinterpret_cast<float2 *>(smem + L::kSlotOff);
    const uint32_t xbar = smem_addr(smem + L::kXbarOff);
    const int tid = threadIdx.x;

    const uint32_t rank = cluster_rank(), csize = cluster_size();
    const int64_t row = blockIdx.x / csize;
    RowView<T> rv(in + row * stride, out + row * stride, cols, vec_store != 0);

    // this block's slice of the row's vectors
    const int64_t per = (rv.nvec + csize - 1) / csize;
    const int64_t s0 = min((int64_t)rank * per, rv.nvec), s1 = min(s0 + per, rv.nvec);
    if (tid == 0) prefetch_span_l2(in + row * stride, s0 * V - rv.head, s1 * V - rv.head, cols);
    pdl_enter();

    if (tid == 0) {
        mbar_init(xbar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(xbar, csize * 8u);  // csize states will arrive
    }
    __syncthreads();
    cluster_arrive_relaxed();  // this block runs and its barrier is armed
    Tile<T, VPT> tile;
    tile.template load<WHOLE>(rv, s0 + tid, THREADS, s1);
    const float2 s = tile.stats();
    float m = s.x, l = s.y;
    block_merge<NW>(m, l, red);
    if (cluster_exchange<NW>(m, l, slots, xbar, rank, csize, wait_ns, starve))
        tile.template scale_store<WHOLE>(rv, s0 + tid, THREADS, s1, out_factor(s.x, m, l));
}

// ---------------------------------------------------------------------------
// path 6: a cluster per row streaming its slices twice (rows of any length)
// ---------------------------------------------------------------------------
// Each of the csize blocks owns a slice of the row, of any length.  Pass 1
// streams the slice tile by tile into one (s, l) state; the states are
// exchanged inside the cluster (distributed shared memory, nothing written to
// global memory); pass 2 streams the slice again and writes
// y = 2^(x log2 e - S) / L.  Three element crossings, the re-read usually
// served by L2 (a block reads its slice again right after pass 1), and no
// scratch: the long-row fallback that allocates nothing.
template <typename T, int THREADS, int VPT, bool WHOLE>
__global__ void __launch_bounds__(THREADS, (THREADS >= 1024 ? 1 : 1024 / THREADS))
    k_cluster_stream(const T *in, T *out, int64_t rows, int64_t cols, int64_t stride, int vec_store,
                     int64_t wait_ns, int starve) {
    if (!explicit_cluster()) {  // launched without clusters: touch no cluster state
        pdl_enter();
        if (threadIdx.x == 0) atomicOr(&g_error_word, kErrNotCluster);
        return;
    }
    constexpr int V = Elem<T>::kVec;
    constexpr int NW = THREADS / 32;
    constexpr int64_t kTile = (int64_t)THREADS * VPT;
    using L = ClusterSmem<THREADS>;
    extern __shared__ __align__(128) unsigned char smem[];
    float2 *red = reinterpret_cast<float2 *>(smem + L::kRedOff);
    float2 *slots = reinterpret_cast<float2 *>(smem + L::kSlotOff);
    const uint32_t xbar = smem_addr(smem + L::kXbarOff);
    const int tid = threadIdx.x;

    const uint32_t rank = cluster_rank(), csize = cluster_size();
    const int64_t row = blockIdx.x / csize;
    RowView<T> rv(in + row * stride, out + row * stride, cols, vec_store != 0);
    const int64_t per = (rv.nvec + csize - 1) / csize;
    const int64_t s0 = min((int64_t)rank * per, rv.nvec), s1 = min(s0 + per, rv.nvec);
    // the first kAhead + 1 tiles of the slice start moving into L2 before the
    // launch-overlap wait; pass 1 then keeps kAhead tiles ahead of its loads
    // (hints: a prefetch cannot change what a later load returns).  A block
    // holds one tile in registers at a time, so without them its bytes in
    // flight, not HBM, bound a slice of many tiles.
    constexpr int64_t kAhead = 2;
    if (tid == 0)
        prefetch_span_l2(rv.in, s0 * V - rv.head, min(s0 + (kAhead + 1) * kTile, s1) * V - rv.head, cols);
    pdl_enter();

    if (tid == 0) {
        mbar_init(xbar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(xbar, csize * 8u);  // csize states will arrive
    }
    __syncthreads();
    cluster_arrive_relaxed();  // this block runs and its barrier is armed

    // pass 1: the slice's state
    float m = -INFINITY, l = 0.f;
    for (int64_t t0 = s0; t0 < s1; t0 += kTile) {
        const int64_t p0 = t0 + (kAhead + 1) * kTile;
        if (tid == 0 && p0 < s1) prefetch_span_l2(rv.in, p0 * V - rv.head, min(p0 + kTile, s1) * V - rv.head, cols);
        Tile<T, VPT> tile;
        tile.template load<WHOLE>(rv, t0 + tid, THREADS, s1);
        const float2 st = tile.stats();
        const float M = fmaxf(m, st.x);
        l = rescale(l, m, M) + rescale(st.y, st.x, M);
        m = M;
    }
    block_merge<NW>(m, l, red);
    if (!cluster_exchange<NW>(m, l, slots, xbar, rank, csize, wait_ns, starve)) return;

    // pass 2: re-read and write (m is the row's S)
    const float inv = m == -INFINITY ? __int_as_float(0x7fc00000) : 1.f / l;
    for (int64_t t0 = s0; t0 < s1; t0 += kTile) {
        Tile<T, VPT> tile;
        tile.template load<WHOLE>(rv, t0 + tid, THREADS, s1);
        tile.template shift_store<WHOLE>(rv, t0 + tid, THREADS, s1, m, inv);
    }
}

// ---------------------------------------------------------------------------
// path 4: rows split over the grid (two passes, states in scratch)
// ---------------------------------------------------------------------------
// L2 prefetch of this block's first chunk (one thread), ahead of pdl_enter.
template <typename T>
__device__ __forceinline__ void prefetch_first_chunk(const T *in, int64_t rows, int64_t cols, int64_t stride,
                                                     int64_t chunks, int64_t chunk_vecs) {
    constexpr int V = Elem<T>::kVec;
    if (threadIdx.x != 0 || (int64_t)blockIdx.x >= rows * chunks) return;
    const int64_t row = blockIdx.x / chunks, k = blockIdx.x - row * chunks;
    const RowView<T> rv(in + row * stride, nullptr, cols, false);
    prefetch_span_l2(rv.in, k * chunk_vecs * V - rv.head, (k + 1) * chunk_vecs * V - rv.head, cols);
}

template <typename T, int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS) k_split_stats(const T *in, int64_t rows, int64_t cols, int64_t stride,
                                                         int64_t chunks, int64_t chunk_vecs, float2 *part) {
    prefetch_first_chunk(in, rows, cols, stride, chunks, chunk_vecs);
    pdl_enter();
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
            const float2 s = tile.stats();
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
    prefetch_first_chunk(in, rows, cols, stride, chunks, chunk_vecs);
    pdl_enter();
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
            tile.shift_store(rv, t0 + threadIdx.x, THREADS, c1, shift, inv);
        }
    }
}

// ---------------------------------------------------------------------------
// path 8: a few very long rows over the whole grid, the per-chunk states kept
// in the output row itself (out != in; two launches, nothing allocated)
// ---------------------------------------------------------------------------
// Chunk k (of `chunks`) of a row covers vectors [k chunk_vecs, (k + 1)
// chunk_vecs), the last chunk also the rest of the row.  The row's state
// region is the start of its output row, from its first 4-byte aligned byte:
// one 8-byte slot per chunk (the chunk's (s, l) as the bit patterns of two
// floats), then a 32-bit counter.  The planner keeps the region inside the
// row.
//
// k_grid_stats: each block streams a chunk into its state, writes the slot,
// and the block of chunk 0 zeroes the counter.
// k_grid_apply (after k_grid_stats has completed, griddepcontrol.wait):
// each block reads every slot of its row, folds them into the row's state,
// counts itself on the counter (fence, then atomicAdd) and writes its chunk
// but the vectors that cover the region.  The block that counts last knows
// every block of the row has read the slots: it writes the region's vectors
// (fence, then re-read from `in`).  No block waits on another.
template <typename T>
struct GridStates {
    uint32_t *w;  // the region: slot k = w[2k], w[2k + 1]; the counter = w[2 chunks]
    __device__ __forceinline__ explicit GridStates(T *out_row)
        : w(reinterpret_cast<uint32_t *>((reinterpret_cast<uintptr_t>(out_row) + 3) & ~(uintptr_t)3)) {}
    __device__ __forceinline__ void put(int64_t k, float2 st) const {
        w[2 * k] = __float_as_uint(st.x);
        w[2 * k + 1] = __float_as_uint(st.y);
    }
    // through L2 (the slots were written by the previous launch)
    __device__ __forceinline__ float2 get(int64_t k) const {
        return make_float2(__uint_as_float(__ldcg(w + 2 * k)), __uint_as_float(__ldcg(w + 2 * k + 1)));
    }
    __device__ __forceinline__ unsigned int *counter(int64_t chunks) const { return w + 2 * chunks; }
    // vectors [0, r) of the row view `rv` (the input's vector geometry) cover
    // the region's columns
    __device__ __forceinline__ int64_t region_vecs(const RowView<T> &rv, const T *out_row, int64_t chunks) const {
        const int64_t bytes = (int64_t)(reinterpret_cast<uintptr_t>(w) - reinterpret_cast<uintptr_t>(out_row)) +
                              8 * chunks + 4;
        const int64_t n = (bytes + (int64_t)sizeof(T) - 1) / (int64_t)sizeof(T);
        return (rv.head + n + Elem<T>::kVec - 1) / Elem<T>::kVec;
    }
};

__device__ __forceinline__ void grid_chunk(int64_t k, int64_t chunks, int64_t chunk_vecs, int64_t nvec,
                                           int64_t &c0, int64_t &c1) {
    c0 = min(k * chunk_vecs, nvec);
    c1 = k == chunks - 1 ? nvec : min(c0 + chunk_vecs, nvec);
}

template <typename T, int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS) k_grid_stats(const T *in, T *out, int64_t rows, int64_t cols,
                                                        int64_t stride, int64_t chunks, int64_t chunk_vecs) {
    prefetch_first_chunk(in, rows, cols, stride, chunks, chunk_vecs);
    pdl_enter();
    constexpr int NW = THREADS / 32;
    constexpr int64_t kTile = (int64_t)THREADS * VPT;
    __shared__ float2 red[2][NW];
    int parity = 0;
    const int64_t units = rows * chunks;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x, parity ^= 1) {
        const int64_t row = u / chunks, k = u - row * chunks;
        RowView<T> rv(in + row * stride, out + row * stride, cols, false);
        int64_t c0, c1;
        grid_chunk(k, chunks, chunk_vecs, rv.nvec, c0, c1);
        float m = -INFINITY, l = 0.f;
        for (int64_t t0 = c0; t0 < c1; t0 += kTile) {
            Tile<T, VPT> tile;
            tile.load(rv, t0 + threadIdx.x, THREADS, c1);
            const float2 st = tile.stats();
            const float M = fmaxf(m, st.x);
            l = rescale(l, m, M) + rescale(st.y, st.x, M);
            m = M;
        }
        block_merge<NW>(m, l, red[parity]);
        if (threadIdx.x == 0) {
            const GridStates<T> gs(out + row * stride);
            gs.put(k, make_float2(m, l));
            if (k == 0) *gs.counter(chunks) = 0u;
        }
    }
}

template <typename T, int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS, VPT == 4 ? 1024 / THREADS : 1)
    k_grid_apply(const T *in, T *out, int64_t rows, int64_t cols, int64_t stride, int64_t chunks,
                 int64_t chunk_vecs, int vec_store) {
    prefetch_first_chunk(in, rows, cols, stride, chunks, chunk_vecs);
    pdl_enter();
    constexpr int NW = THREADS / 32;
    constexpr int64_t kTile = (int64_t)THREADS * VPT;
    __shared__ float2 red[2][NW];
    __shared__ int last_flag[2];
    int parity = 0;
    const int64_t units = rows * chunks;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x, parity ^= 1) {
        const int64_t row = u / chunks, k = u - row * chunks;
        T *orow = out + row * stride;
        RowView<T> rv(in + row * stride, orow, cols, vec_store != 0);
        const GridStates<T> gs(orow);
        int64_t c0, c1;
        grid_chunk(k, chunks, chunk_vecs, rv.nvec, c0, c1);
        const int64_t r = gs.region_vecs(rv, orow, chunks);
        const int64_t s0 = max(c0, r);  // the chunk's first vector past the region
        Tile<T, VPT> tile;
        if (s0 < c1) tile.load(rv, s0 + threadIdx.x, THREADS, c1);  // in flight while the slots are read
        float m = -INFINITY, l = 0.f;
        for (int64_t j = threadIdx.x; j < chunks; j += THREADS) {
            const float2 st = gs.get(j);
            const float M = fmaxf(m, st.x);
            l = rescale(l, m, M) + rescale(st.y, st.x, M);
            m = M;
        }
        block_merge<NW>(m, l, red[parity]);  // every thread's slot reads have returned
        if (threadIdx.x == 0) {
            __threadfence();
            const bool last = atomicAdd(gs.counter(chunks), 1u) == (unsigned int)(chunks - 1);
            if (last) __threadfence();
            last_flag[parity] = last;
        }
        __syncthreads();
        const float shift = m;  // the row's S
        const float inv = m == -INFINITY ? __int_as_float(0x7fc00000) : 1.f / l;
        // the chunk past the region, then (the last block only, once every
        // block of the row has read the slots) the region's vectors
        const int passes = last_flag[parity] ? 2 : 1;
        for (int pass = 0; pass < passes; ++pass) {
            const int64_t a = pass == 0 ? s0 : 0, b = pass == 0 ? c1 : r;
            for (int64_t t0 = a; t0 < b; t0 += kTile) {
                if (pass != 0 || t0 != s0) tile.load(rv, t0 + threadIdx.x, THREADS, b);
                tile.shift_store(rv, t0 + threadIdx.x, THREADS, b, shift, inv);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// path 7: narrow dense rows staged through shared memory
// ---------------------------------------------------------------------------
// Rows of a dense matrix (row stride == cols) too narrow and too misaligned
// for per-row vector access (fp32 rows 39 wide: two of every row's ten
// vectors are partial, and a lane group per row pays its per-row costs on
// every lane) are taken rows_per_span at a time as one contiguous span.  The
// span moves between HBM and shared memory in whole 16-byte vectors -- only
// its two end vectors, which it shares with the neighbouring spans, go
// element by element -- and one thread per row works on the staged floats in
// three sweeps: the max, then e = 2^(x log2 e - s) with its sum (e written
// back), then e / sum.  A thread's rows start cols floats apart, so odd widths
// read shared memory without bank conflicts.
template <typename T>
__global__ void __launch_bounds__(128) k_packed_rows(const T *in, T *out, int64_t rows, int64_t cols,
                                                     int rows_per_span) {
    constexpr int THREADS = 128, V = Elem<T>::kVec;
    extern __shared__ __align__(16) float span[];
    const int64_t total = rows * cols;
    const int head0 = (int)((reinterpret_cast<uintptr_t>(in) & (kVecBytes - 1)) / sizeof(T));
    const uint4 *vin = reinterpret_cast<const uint4 *>(in - head0);
    uint4 *vout = reinterpret_cast<uint4 *>(out - head0);  // out has in's 16-byte phase
    const int64_t nspans = (rows + rows_per_span - 1) / rows_per_span;
    if (threadIdx.x == 0 && (int64_t)blockIdx.x < nspans) {
        const int64_t r0 = (int64_t)blockIdx.x * rows_per_span;
        prefetch_span_l2(in, r0 * cols, min(r0 + rows_per_span, rows) * cols, total);
    }
    pdl_enter();
    for (int64_t sp = blockIdx.x; sp < nspans; sp += gridDim.x) {
        const int64_t r0 = sp * rows_per_span, r1 = min(r0 + rows_per_span, rows);
        const int64_t e0 = r0 * cols, e1 = r1 * cols;
        const int64_t k_lo = (e0 + head0) / V, k_hi = (e1 + head0 + V - 1) / V;
        const int64_t a0 = k_lo * V - head0;  // the element held by span[0]
        // HBM -> shared memory, whole vectors but at the matrix's two ends
        for (int64_t k = k_lo + threadIdx.x; k < k_hi; k += THREADS) {
            const int64_t el = k * V - head0;
            float x[V];
            if (el >= 0 && el + V <= total) {
                Elem<T>::unpack(vin[k], x);
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i) x[i] = (el + i >= 0 && el + i < total) ? Elem<T>::to_f(in[el + i]) : 0.f;
            }
            float4 *d = reinterpret_cast<float4 *>(span + (el - a0));
#pragma unroll
            for (int i = 0; i < V / 4; ++i) d[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
        }
        __syncthreads();
        // one thread per row
        for (int64_t r = r0 + threadIdx.x; r < r1; r += THREADS) {
            float *row = span + (r * cols - a0);
            float m = -INFINITY;
            for (int64_t c = 0; c < cols; ++c) m = fmaxf(m, row[c]);
            const float s = m * kLog2e;
            const float shift = safe_shift(s);
            float l = 0.f;
            for (int64_t c = 0; c < cols; ++c) {
                const float e = ex2(fmaf(row[c], kLog2e, -shift));
                row[c] = e;
                l += e;
            }
            const float f = out_factor(s, s, l);
            for (int64_t c = 0; c < cols; ++c) row[c] *= f;
        }
        __syncthreads();
        // shared memory -> HBM: whole vectors inside the span, its two end
        // vectors element by element (their other elements belong to the
        // neighbouring spans)
        for (int64_t k = k_lo + threadIdx.x; k < k_hi; k += THREADS) {
            const int64_t el = k * V - head0;
            const float *src = span + (el - a0);
            if (el >= e0 && el + V <= e1) {
                vout[k] = Elem<T>::pack(src);
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i)
                    if (el + i >= e0 && el + i < e1) out[el + i] = Elem<T>::from_f(src[i]);
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// scaled, causally masked rows (softmax_fwd_masked)
// ---------------------------------------------------------------------------
// Page "Dissecting Memory Bandwidth & SRAM Tiling in Triton: From GEMM to
// FlashAttention-3", section "Writing the Kernel in OpenAI Triton": scores
// are x * scale and a key after its query is -inf before the softmax.  Row r
// keeps n = mask.kept(r, cols) columns: only those are read (a row view of n
// columns), the row is written in full (a row view of cols columns), the
// masked outputs being 0 -- or NaN when the row itself is NaN (nothing kept,
// or a NaN / +inf among the kept entries), which the row's output factor f
// shows: the zeros are stored while the loads are in flight, and a NaN row
// stores its masked part again.

// The first of the vectors first, first + step, ... that is >= lo.
__device__ __forceinline__ int64_t first_from(int64_t first, int64_t step, int64_t lo) {
    if (first >= lo) return first;
    return first + ((lo - first + step - 1) / step) * step;
}

// Store `value` into every element of vectors first, first + step, ... below
// end (WHOLE: rows of whole vectors, plain 16-byte stores).
template <bool WHOLE, typename T>
__device__ __forceinline__ void fill_vectors(const RowView<T> &row, int64_t first, int64_t step, int64_t end,
                                             float value) {
    float y[Elem<T>::kVec];
#pragma unroll
    for (int i = 0; i < Elem<T>::kVec; ++i) y[i] = value;
    if constexpr (WHOLE) {
        const uint4 w = Elem<T>::pack(y);
        uint4 *q = reinterpret_cast<uint4 *>(row.out);
        for (int64_t v = first; v < end; v += step) q[v] = w;
    } else {
        for (int64_t v = first; v < end; v += step) row.store(v, y);
    }
}

// Load a thread's kept vectors first + j*step of a row view `rl` of the kept
// columns.  16-bit rows: every kept vector as an aligned 16-byte load, the
// elements of a partial last one past the kept part masked to -inf (the
// packed tile's own load).  fp32 rows of whole vectors (WHOLE): every kept
// vector but a last partial one as a plain 16-byte load, the partial one
// element by element.
template <bool WHOLE, int VPT, typename Tl, typename T>
__device__ __forceinline__ void load_kept(Tl &tile, const RowView<T> &rl, int64_t first, int64_t step) {
    if constexpr (sizeof(T) == 2) {
        tile.load(rl, first, step, rl.nvec);
    } else if constexpr (WHOLE) {
        constexpr int V = Elem<T>::kVec;
        const int64_t nw = rl.cols / V;  // whole kept vectors (rows start on 16 bytes)
        tile.template load<true>(rl, first, step, nw);
        if (rl.cols % V != 0) {
#pragma unroll
            for (int j = 0; j < VPT; ++j)
                if (first + j * step == nw) tile.load_one(j, rl, nw);
        }
    } else {
        tile.load(rl, first, step, rl.nvec);
    }
}

template <typename T, int G, int VPT, bool WHOLE>
__global__ void __launch_bounds__(256) k_warp_rows_masked(const T *in, T *out, int64_t rows, int64_t cols,
                                                          int64_t stride, int vec_store, CausalMask mask) {
    const int t = threadIdx.x & (G - 1);
    const int64_t groups_per_block = blockDim.x / G;
    const int64_t row_step = (int64_t)gridDim.x * groups_per_block;
    const int64_t warp_row0 = (int64_t)blockIdx.x * groups_per_block + (threadIdx.x & ~31) / G;
    if (t == 0 && warp_row0 + (threadIdx.x & 31) / G < rows) {
        const int64_t r = warp_row0 + (threadIdx.x & 31) / G;
        prefetch_span_l2(in + r * stride, 0, mask.kept(r, cols), cols);
    }
    pdl_enter();
    for (int64_t base = warp_row0; base < rows; base += row_step) {
        const int64_t row = base + (threadIdx.x & 31) / G;
        const bool active = row < rows;
        const int64_t r = active ? row : 0;
        RowView<T> rl(in + r * stride, out + r * stride, active ? mask.kept(row, cols) : 0, vec_store != 0);
        RowView<T> rs(in + r * stride, out + r * stride, cols, vec_store != 0);
        Tile<T, VPT> tile;
        load_kept<WHOLE, VPT>(tile, rl, t, G);
        // the masked outputs do not depend on the loads: their zeros go out
        // while the loads are in flight
        const int64_t fill0 = first_from(t, G, rl.nvec);
        if (active) fill_vectors<WHOLE>(rs, fill0, G, rs.nvec, 0.f);
        const float2 s = tile.stats(mask.k, live_slots(t, G, rl.nvec, VPT));
        float m = s.x, l = s.y;
        group_merge<G>(m, l);
        if (active) {
            const float f = out_factor(s.x, m, l);
            tile.template scale_store<WHOLE>(rs, t, G, rl.nvec, f);
            if (isnan(f)) fill_vectors<WHOLE>(rs, fill0, G, rs.nvec, f);  // a NaN row
        }
    }
}

template <typename T, int THREADS, int VPT, bool WHOLE>
__device__ __forceinline__ void cta_rows_masked_body(const T *in, T *out, int64_t rows, int64_t cols,
                                                     int64_t stride, int vec_store, const CausalMask &mask) {
    constexpr int NW = THREADS / 32;
    __shared__ float2 red[2][NW];
    if (threadIdx.x == 0 && blockIdx.x < rows)
        prefetch_span_l2(in + blockIdx.x * stride, 0, mask.kept(blockIdx.x, cols), cols);
    pdl_enter();
    int parity = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, parity ^= 1) {
        RowView<T> rl(in + row * stride, out + row * stride, mask.kept(row, cols), vec_store != 0);
        RowView<T> rs(in + row * stride, out + row * stride, cols, vec_store != 0);
        Tile<T, VPT> tile;
        load_kept<WHOLE, VPT>(tile, rl, threadIdx.x, THREADS);
        const int64_t fill0 = first_from(threadIdx.x, THREADS, rl.nvec);
        fill_vectors<WHOLE>(rs, fill0, THREADS, rs.nvec, 0.f);  // while the loads are in flight
        const float2 s = tile.stats(mask.k, live_slots(threadIdx.x, THREADS, rl.nvec, VPT));
        float m = s.x, l = s.y;
        block_merge<NW>(m, l, red[parity]);
        const float f = out_factor(s.x, m, l);
        tile.template scale_store<WHOLE>(rs, threadIdx.x, THREADS, rl.nvec, f);
        if (isnan(f)) fill_vectors<WHOLE>(rs, fill0, THREADS, rs.nvec, f);  // a NaN row
    }
}

template <typename T, int THREADS, int VPT, bool WHOLE>
__global__ void __launch_bounds__(THREADS) k_cta_rows_masked(const T *in, T *out, int64_t rows, int64_t cols,
                                                             int64_t stride, int vec_store, CausalMask mask) {
    cta_rows_masked_body<T, THREADS, VPT, WHOLE>(in, out, rows, cols, stride, vec_store, mask);
}

template <typename T, int THREADS, int VPT, bool WHOLE>
__global__ void __launch_bounds__(THREADS, 1024 / THREADS)
    k_cta_rows_masked_wide(const T *in, T *out, int64_t rows, int64_t cols, int64_t stride, int vec_store,
                           CausalMask mask) {
    cta_rows_masked_body<T, THREADS, VPT, WHOLE>(in, out, rows, cols, stride, vec_store, mask);
}

// The streaming cluster of path 6 on masked rows: every block owns a slice
// of the full row; it reads only the kept part of its slice, in both passes.
template <typename T, int THREADS, int VPT, bool WHOLE>
__global__ void __launch_bounds__(THREADS, (THREADS >= 1024 ? 1 : 1024 / THREADS))
    k_cluster_stream_masked(const T *in, T *out, int64_t rows, int64_t cols, int64_t stride, int vec_store,
                            int64_t wait_ns, int starve, CausalMask mask) {
    if (!explicit_cluster()) {  // launched without clusters: touch no cluster state
        pdl_enter();
        if (threadIdx.x == 0) atomicOr(&g_error_word, kErrNotCluster);
        return;
    }
    constexpr int V = Elem<T>::kVec;
    constexpr int NW = THREADS / 32;
    constexpr int64_t kTile = (int64_t)THREADS * VPT;
    using L = ClusterSmem<THREADS>;
    extern __shared__ __align__(128) unsigned char smem[];
    float2 *red = reinterpret_cast<float2 *>(smem + L::kRedOff);
    float2 *slots = reinterpret_cast<float2 *>(smem + L::kSlotOff);
    const uint32_t xbar = smem_addr(smem + L::kXbarOff);
    const int tid = threadIdx.x;

    const uint32_t rank = cluster_rank(), csize = cluster_size();
    const int64_t row = blockIdx.x / csize;
    RowView<T> rl(in + row * stride, out + row * stride, mask.kept(row, cols), vec_store != 0);
    RowView<T> rs(in + row * stride, out + row * stride, cols, vec_store != 0);
    const int64_t per = (rs.nvec + csize - 1) / csize;
    const int64_t s0 = min((int64_t)rank * per, rs.nvec), s1 = min(s0 + per, rs.nvec);
    const int64_t k1 = min(s1, rl.nvec);  // this slice's kept vectors: [s0, k1)
    if (tid == 0) prefetch_span_l2(rl.in, s0 * V - rl.head, min(s0 + kTile, k1) * V - rl.head, rl.cols);
    pdl_enter();

    if (tid == 0) {
        mbar_init(xbar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(xbar, csize * 8u);
    }
    __syncthreads();
    cluster_arrive_relaxed();
    const int64_t fill0 = first_from(s0 + tid, THREADS, k1);
    fill_vectors<WHOLE>(rs, fill0, THREADS, s1, 0.f);  // the masked part of the slice

    float m = -INFINITY, l = 0.f;
    for (int64_t t0 = s0; t0 < k1; t0 += kTile) {
        Tile<T, VPT> tile;
        tile.load(rl, t0 + tid, THREADS, k1);
        const float2 st = tile.stats(mask.k, live_slots(t0 + tid, THREADS, k1, VPT));
        const float M = fmaxf(m, st.x);
        l = rescale(l, m, M) + rescale(st.y, st.x, M);
        m = M;
    }
    block_merge<NW>(m, l, red);
    if (!cluster_exchange<NW>(m, l, slots, xbar, rank, csize, wait_ns, starve)) return;

    const float inv = m == -INFINITY ? __int_as_float(0x7fc00000) : 1.f / l;
    for (int64_t t0 = s0; t0 < k1; t0 += kTile) {
        Tile<T, VPT> tile;
        tile.load(rl, t0 + tid, THREADS, k1);
        tile.template shift_store<WHOLE>(rs, t0 + tid, THREADS, k1, m, inv, mask.k);
    }
    if (isnan(inv)) fill_vectors<WHOLE>(rs, fill0, THREADS, s1, inv);  // a NaN row
}

}  // namespace mbrs
