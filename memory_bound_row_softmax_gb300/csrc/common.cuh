// common.cuh -- device building blocks shared by the row-softmax kernels.
//
// Every kernel computes, per row, the numerically stable softmax
//     y_c = exp(x_c - m) / l,   m = max_c x_c,   l = sum_c exp(x_c - m)
// (page "Dissecting Memory Bandwidth & SRAM Tiling in Triton", section "The
// Mathematical Remedy: Online Softmax Tiling") with one read and one write of
// each element (page "fused-softmax-roofline").
//
// Per-thread state.  A thread holds its elements in registers, takes its own
// max m_t, turns its elements into e_c = exp(x_c - m_t) at once and sums them
// into l_t.  The (m_t, l_t) pairs of all threads of a row are then combined
// with the two-state merge rule of the same section,
//     m = max(m1, m2),   l = l1 exp(m1 - m) + l2 exp(m2 - m),
// and each thread finally scales its e_c by exp(m_t - m) / l.  This needs one
// exp per element and ONE cross-thread reduction per row (instead of a max
// reduction followed by a sum reduction), which matters most where the row
// spans the warps of a block or the blocks of a cluster.
//
// exp is computed as 2^(x log2 e - s) with the PTX instruction
// ex2.approx.ftz.f32 (relative error about 2^-22), where s = fl(m log2 e) is
// the shift rounded once to fp32.  States are carried in that base-2 form,
// (s, l) with l = sum 2^(x log2 e - s), and merged as
//     S = max(s1, s2),   l = l1 2^(s1 - S) + l2 2^(s2 - S),
// so every element of a row ends up scaled by the same 2^(-S): the rounding
// of the shift cancels in the ratio instead of differing from thread to thread
// (with |m| near 100 a per-thread rounding would cost ~5e-6 relative).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mbrs {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)
constexpr int kVecBytes = 16;                  // one 128-bit access

// ---------------------------------------------------------------------------
// element types
// ---------------------------------------------------------------------------
template <typename T> struct Elem;

template <> struct Elem<float> {
    static constexpr int kVec = 4;  // elements per 16-byte vector
    static constexpr uint32_t kNegInfBits = 0xff800000u;
    __device__ static __forceinline__ float to_f(float v) { return v; }
    __device__ static __forceinline__ float from_f(float v) { return v; }
    __device__ static __forceinline__ void unpack(const uint4 &r, float *x) {
        x[0] = __uint_as_float(r.x);
        x[1] = __uint_as_float(r.y);
        x[2] = __uint_as_float(r.z);
        x[3] = __uint_as_float(r.w);
    }
    __device__ static __forceinline__ uint4 pack(const float *y) {
        return make_uint4(__float_as_uint(y[0]), __float_as_uint(y[1]), __float_as_uint(y[2]),
                          __float_as_uint(y[3]));
    }
};

template <> struct Elem<__half> {
    static constexpr int kVec = 8;
    static constexpr uint16_t kNegInfBits = 0xfc00;
    __device__ static __forceinline__ float to_f(__half v) { return __half2float(v); }
    __device__ static __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
    __device__ static __forceinline__ float2 pair(uint32_t w) {
        __half2 h = *reinterpret_cast<const __half2 *>(&w);
        return __half22float2(h);
    }
    __device__ static __forceinline__ uint32_t unpair(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
    __device__ static __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
        __half2 r = __hmax2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
        return *reinterpret_cast<const uint32_t *>(&r);
    }
    __device__ static __forceinline__ void unpack(const uint4 &r, float *x) {
        float2 p;
        p = pair(r.x); x[0] = p.x; x[1] = p.y;
        p = pair(r.y); x[2] = p.x; x[3] = p.y;
        p = pair(r.z); x[4] = p.x; x[5] = p.y;
        p = pair(r.w); x[6] = p.x; x[7] = p.y;
    }
    __device__ static __forceinline__ uint4 pack(const float *y) {
        return make_uint4(unpair(y[0], y[1]), unpair(y[2], y[3]), unpair(y[4], y[5]),
                          unpair(y[6], y[7]));
    }
};

template <> struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
    static constexpr uint16_t kNegInfBits = 0xff80;
    __device__ static __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ static __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
    __device__ static __forceinline__ float2 pair(uint32_t w) {
        // bf16 -> f32 is exact: the bf16 bits are the top half of the f32
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    __device__ static __forceinline__ uint32_t unpair(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
    __device__ static __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
        __nv_bfloat162 r = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&a),
                                   *reinterpret_cast<const __nv_bfloat162 *>(&b));
        return *reinterpret_cast<const uint32_t *>(&r);
    }
    __device__ static __forceinline__ void unpack(const uint4 &r, float *x) {
        float2 p;
        p = pair(r.x); x[0] = p.x; x[1] = p.y;
        p = pair(r.y); x[2] = p.x; x[3] = p.y;
        p = pair(r.z); x[4] = p.x; x[5] = p.y;
        p = pair(r.w); x[6] = p.x; x[7] = p.y;
    }
    __device__ static __forceinline__ uint4 pack(const float *y) {
        return make_uint4(unpair(y[0], y[1]), unpair(y[2], y[3]), unpair(y[4], y[5]),
                          unpair(y[6], y[7]));
    }
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Low 32 bits of the global nanosecond timer (wraps every 4.29 s; differences
// taken modulo 2^32 are right for intervals shorter than that).
__device__ __forceinline__ uint32_t global_timer_lo() {
    uint32_t t;
    asm volatile("mov.u32 %0, %%globaltimer_lo;" : "=r"(t));
    return t;
}

// Programmatic dependent launch.  griddepcontrol.wait returns once the grid
// this one depends on (the previous kernel in the stream, when this grid was
// launched with programmatic stream serialisation; otherwise nothing) has
// completed and its memory operations are visible.  Every kernel calls this
// before its first global-memory access, then lets the next grid in the stream
// be scheduled: that grid waits the same way before it touches memory.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2 prefetch hints.  A prefetch does not change what any later load
// returns, so a kernel may issue them before griddepcontrol.wait: with launch
// overlap its input starts moving from HBM into L2 while the previous kernel
// is still finishing.  Only the 16-byte-aligned interior of elements
// [e0, e1) of a row of `cols` elements (clipped to the row) is prefetched, so
// no byte outside the row is named.
constexpr uintptr_t kPrefetchPiece = 65536;
__device__ __forceinline__ void prefetch_l2(uintptr_t addr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(addr), "r"(bytes) : "memory");
}
template <typename T>
__device__ __forceinline__ void prefetch_span_l2(const T *row, int64_t e0, int64_t e1, int64_t cols) {
    e0 = max(e0, (int64_t)0);
    e1 = min(e1, cols);
    if (e1 <= e0) return;
    const uintptr_t a = ((uintptr_t)(row + e0) + 15) & ~(uintptr_t)15;
    const uintptr_t e = (uintptr_t)(row + e1) & ~(uintptr_t)15;
    for (uintptr_t q = a; q < e; q += kPrefetchPiece) prefetch_l2(q, (uint32_t)min(e - q, kPrefetchPiece));
}

// mbarrier (shared::cta) -- arrival/transaction barrier the TMA engine completes.
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for phase `parity` of an mbarrier: gives up after limit_ns of
// global time and returns false.  Never spins without a bound.
// The timer is read 32 bits wide (two fewer live registers in the waits that
// sit beside register-held tiles), so limit_ns is capped at 2^31 ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, int64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint32_t limit = (uint32_t)min(limit_ns, (int64_t)0x7fffffff);
    const uint32_t t0 = global_timer_lo();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_lo() - t0 > limit) return false;
    }
    return false;
}

// 1-D TMA bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Order this thread's earlier generic-proxy accesses to shared memory before
// later async-proxy (TMA) accesses to it.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// thread-block cluster
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// True when this grid was launched with explicit cluster dimensions.
__device__ __forceinline__ bool explicit_cluster() {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmov.pred p, %%is_explicit_cluster;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r));
    return r != 0;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// Asynchronous store of two floats into a peer block's shared memory; the 8
// bytes count against the peer's mbarrier at remote_bar (complete_tx).
__device__ __forceinline__ void st_async_f2(uint32_t remote_addr, float a, float b, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
                     remote_addr),
                 "f"(a), "f"(b), "r"(remote_bar)
                 : "memory");
}
__device__ __forceinline__ void st_cluster_f2(uint32_t addr, float a, float b) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}


// ---------------------------------------------------------------------------
// (s, l) states, s = fl(max * log2 e)
// ---------------------------------------------------------------------------
// The shift an element uses: an empty state (s = -inf) shifts by 0 so that
// its (all -inf) entries give 2^-inf = 0 instead of NaN.
__device__ __forceinline__ float safe_shift(float s) { return s == -INFINITY ? 0.f : s; }

// l taken from shift s to shift S >= s (0 for an empty state).
__device__ __forceinline__ float rescale(float l, float s, float S) {
    return s == -INFINITY ? 0.f : l * ex2(s - S);
}

// Merge the states of the `width` lanes of each aligned lane group (width a
// power of two <= 32).  All 32 lanes must call it.
template <int WIDTH>
__device__ __forceinline__ void group_merge(float &m, float &l) {
    float M = m;
#pragma unroll
    for (int o = WIDTH / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = rescale(l, m, M);
#pragma unroll
    for (int o = WIDTH / 2; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    m = M;
    l = L;
}

// The final per-thread factor: e_c * factor = 2^(x_c log2 e - S) / L.  A row
// with no finite max (every entry -inf) gives NaN, as does a NaN or +inf
// entry (L NaN).
__device__ __forceinline__ float out_factor(float s_t, float S, float L) {
    if (S == -INFINITY) return __int_as_float(0x7fc00000);
    return rescale(1.f, s_t, S) * (1.f / L);
}

// ---------------------------------------------------------------------------
// row geometry: a row is covered by 16-byte aligned vectors
// ---------------------------------------------------------------------------
// A row starting at element pointer p has `head` = (address mod 16) / elem
// elements in front of it inside its first aligned vector.  Vector v covers
// the row's columns [v*V - head, v*V - head + V); the row needs
// nvec = ceil((head + cols) / V) vectors.  Only the first and the last vector
// can be partial; those are read and written element by element so that no
// access leaves the row.
template <typename T>
struct RowView {
    static constexpr int V = Elem<T>::kVec;
    const T *in;   // row start (input)
    T *out;        // row start (output)
    int head;      // elements before the row start in its first vector
    int tail;      // elements of the row in its last vector (V when that vector is whole)
    int64_t cols;
    int64_t nvec;
    bool vec_store;  // out has the same 16-byte phase as in

    __device__ __forceinline__ RowView(const T *in_row, T *out_row, int64_t cols_, bool vec_store_)
        : in(in_row), out(out_row), cols(cols_), vec_store(vec_store_) {
        head = (int)((reinterpret_cast<uintptr_t>(in_row) & (kVecBytes - 1)) / sizeof(T));
        nvec = (head + cols + V - 1) / V;
        tail = (int)(head + cols - (nvec - 1) * V);
    }
    // The row's vectors as aligned 16-byte words: vector v is vec_in()[v].
    // Loading a whole aligned vector that holds at least one element of the
    // row cannot fault, also for the row's partial end vectors (an aligned
    // 16-byte block never straddles a page); their elements outside the row
    // must then be masked.  vec_out() is only meaningful with vec_store.
    __device__ __forceinline__ const uint4 *vec_in() const { return reinterpret_cast<const uint4 *>(in - head); }
    __device__ __forceinline__ uint4 *vec_out() const { return reinterpret_cast<uint4 *>(out - head); }

    __device__ __forceinline__ bool full(int64_t v) const {
        const int64_t p = v * V;
        return p >= head && p + V <= head + cols;
    }
    // Load vector v (must be < nvec) as floats; columns outside the row read -inf.
    __device__ __forceinline__ void load(int64_t v, float *x) const {
        const int64_t c0 = v * V - head;
        if (full(v)) {
            Elem<T>::unpack(*reinterpret_cast<const uint4 *>(in + c0), x);
        } else {
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int64_t c = c0 + i;
                x[i] = (c >= 0 && c < cols) ? Elem<T>::to_f(in[c]) : -INFINITY;
            }
        }
    }
    // Load vector v as raw 16-byte storage; for 16-bit types, columns outside
    // the row hold the -inf bit pattern.
    __device__ __forceinline__ uint4 load_raw(int64_t v) const {
        const int64_t c0 = v * V - head;
        if (full(v)) return *reinterpret_cast<const uint4 *>(in + c0);
        static_assert(sizeof(T) == 2, "raw partial vectors are for 16-bit types");
        const uint16_t ninf = Elem<T>::kNegInfBits;
        const uint16_t *src = reinterpret_cast<const uint16_t *>(in);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t ca = c0 + 2 * k, cb = ca + 1;
            const uint32_t a = (ca >= 0 && ca < cols) ? src[ca] : ninf;
            const uint32_t b = (cb >= 0 && cb < cols) ? src[cb] : ninf;
            w[k] = a | (b << 16);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    // Store vector v's results; only columns inside the row are written.
    __device__ __forceinline__ void store(int64_t v, const float *y) const {
        const int64_t c0 = v * V - head;
        if (vec_store && full(v)) {
            *reinterpret_cast<uint4 *>(out + c0) = Elem<T>::pack(y);
        } else {
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int64_t c = c0 + i;
                if (c >= 0 && c < cols) out[c] = Elem<T>::from_f(y[i]);
            }
        }
    }
};

// Tiles of rows made of whole 16-byte vectors only (WHOLE = true: in and out
// 16-byte aligned, row stride and width multiples of 16 bytes, decided by the
// host for the whole call): a thread's vectors first + j*step (j < VPT) move
// as plain 16-byte accesses at constant offsets, with no edge test; those with
// j*step >= whole_fit(first, end) lie past the tile's end.
// How many of a tile's vectors first + j*step (j < vpt) lie below end.
__device__ __forceinline__ int live_slots(int64_t first, int64_t step, int64_t end, int vpt) {
    if (first >= end) return 0;
    const int64_t n = (end - first + step - 1) / step;
    return n < vpt ? (int)n : vpt;
}

__device__ __forceinline__ int whole_fit(int64_t first, int64_t end) {
    return (int)max(min(end - first, (int64_t)0x7fffffff), (int64_t)0);
}

// Bit mask of the 16-bit elements a <= i < b (0 <= a, b <= 4) of a 64-bit word.
__device__ __forceinline__ uint64_t elems64(int a, int b) {
    const uint64_t below_b = b >= 4 ? ~0ull : (1ull << (16 * b)) - 1ull;
    const uint64_t from_a = a >= 4 ? 0ull : ~0ull << (16 * a);
    return below_b & from_a;
}

// The 16-bit elements i of a packed vector with lo <= i < hi (0 <= lo, hi <=
// 8), the others replaced by the bit pattern ninf: one bit select per word
// under a mask built with shifts.
__device__ __forceinline__ uint4 keep_range16(const uint4 &r, int lo, int hi, uint32_t ninf) {
    const uint64_t m0 = elems64(min(lo, 4), min(hi, 4));
    const uint64_t m1 = elems64(max(lo - 4, 0), max(hi - 4, 0));
    const uint32_t n = ninf * 0x10001u;
    const uint32_t k0 = (uint32_t)m0, k1 = (uint32_t)(m0 >> 32), k2 = (uint32_t)m1, k3 = (uint32_t)(m1 >> 32);
    return make_uint4((r.x & k0) | (n & ~k0), (r.y & k1) | (n & ~k1), (r.z & k2) | (n & ~k2),
                      (r.w & k3) | (n & ~k3));
}

// Store the 16-bit elements lo <= i < hi (0 <= lo < hi <= 8) of the packed
// vector w into the aligned 16-byte word at dst, as naturally aligned pieces
// of 2, 4 and 8 bytes: first up to the word's 8-byte boundary, then down from
// it.  The word's other elements belong to a neighbouring row and are not
// touched.
__device__ __forceinline__ void store_range16(uint4 *dst, const uint4 &w, int lo, int hi) {
    const uint64_t h0 = (uint64_t)w.x | ((uint64_t)w.y << 32), h1 = (uint64_t)w.z | ((uint64_t)w.w << 32);
    char *const b = reinterpret_cast<char *>(dst);
    const auto half = [&](int k) { return k < 4 ? h0 : h1; };
    const auto st2 = [&](int k) {
        *reinterpret_cast<uint16_t *>(b + 2 * k) = (uint16_t)(half(k) >> (16 * (k & 3)));
    };
    const auto st4 = [&](int k) {
        *reinterpret_cast<uint32_t *>(b + 2 * k) = (uint32_t)(half(k) >> (16 * (k & 3)));
    };
    const auto st8 = [&](int k) { *reinterpret_cast<uint64_t *>(b + 2 * k) = half(k); };
    int i = lo;
    if ((i & 1) && i < hi) st2(i++);
    if ((i & 2) && i + 2 <= hi) { st4(i); i += 2; }
    if ((i & 4) && i + 4 <= hi) { st8(i); i += 4; }
    if (i + 4 <= hi) { st8(i); i += 4; }
    if (i + 4 <= hi) { st8(i); i += 4; }
    if (i + 2 <= hi) { st4(i); i += 2; }
    if (i < hi) st2(i);
}

// Store a tile's results: for vectors first + j*step < end, val(j, y) fills
// the V floats of vector j, rounded once to T on the way out.
template <typename T, int VPT, bool WHOLE, typename F>
__device__ __forceinline__ void tile_store(const RowView<T> &row, int64_t first, int64_t step, int64_t end,
                                           F &&val) {
    constexpr int V = Elem<T>::kVec;
    if constexpr (WHOLE) {
        uint4 *q = reinterpret_cast<uint4 *>(row.out) + first;
        const int fit = whole_fit(first, end);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            if (j * step < fit) {
                float y[V];
                val(j, y);
                q[j * step] = Elem<T>::pack(y);
            }
        }
    } else if constexpr (sizeof(T) == 2) {
        // interior vectors at constant offsets from the row's aligned base;
        // the row's two partial end vectors as naturally aligned pieces
        // (store_range16), or element by element when out has another phase
        uint4 *q = row.vec_out() + first;
        const int fit = whole_fit(first, end);
        // slot offsets (from `first`) of the row's partial first / last vector, -1 if none
        const int64_t head_slot = (first == 0 && row.head != 0) ? 0 : -1;
        const int64_t tail_slot = row.tail < V ? row.nvec - 1 - first : -1;
        if (!row.vec_store) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                if (j * step < fit) {
                    float y[V];
                    val(j, y);
                    row.store(first + (int64_t)j * step, y);
                }
            }
            return;
        }
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int64_t o = (int64_t)j * step;
            if (o < fit && o != head_slot && o != tail_slot) {
                float y[V];
                val(j, y);
                q[o] = Elem<T>::pack(y);
            }
        }
        // the partial end vectors last (at most two slots of one thread each)
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int64_t o = (int64_t)j * step;
            if (o < fit && (o == head_slot || o == tail_slot)) {
                float y[V];
                val(j, y);
                store_range16(q + o, Elem<T>::pack(y), o == head_slot ? row.head : 0,
                              o == tail_slot ? row.tail : V);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int64_t v = first + j * step;
            if (v < end) {
                float y[V];
                val(j, y);
                row.store(v, y);
            }
        }
    }
}

// A thread's tile of VPT vectors.  Two forms share one interface:
//   FloatTile   the elements widened to fp32 (fp32 data: no extra registers);
//               stats() overwrites them with e = 2^(x log2 e - s_t).
//   PackedTile  the raw 16-bit storage (half the registers of FloatTile for
//               fp16/bf16); stats() overwrites it with the exponentials
//               rounded to fp16 pairs.
// Interface: set(j, raw) / set_empty(j) / load_one(j, row, v) /
// load<WHOLE>(row, first, step, end);
// stats(k = log2 e) -> (s_t, l_t); values(j, f, y): y = e * f for vector j;
// values_shift(j, shift, f, y, k): y = 2^(x k - shift) * f (inputs only,
// before stats()); scale_store<WHOLE>(row, first, step, end, f);
// shift_store<WHOLE>(row, first, step, end, shift, f) (inputs only).
template <typename T, int VPT>
struct FloatTile {
    static constexpr int V = Elem<T>::kVec;
    float x[VPT][V];

    __device__ __forceinline__ void set(int j, const uint4 &raw) { Elem<T>::unpack(raw, x[j]); }
    __device__ __forceinline__ void load_one(int j, const RowView<T> &row, int64_t v) { row.load(v, x[j]); }
    __device__ __forceinline__ void set_empty(int j) {
#pragma unroll
        for (int i = 0; i < V; ++i) x[j][i] = -INFINITY;
    }
    // load vectors first + j*step (j < VPT) of a row, -inf past `end`
    template <bool WHOLE = false>
    __device__ __forceinline__ void load(const RowView<T> &row, int64_t first, int64_t step, int64_t end) {
        if constexpr (WHOLE) {
            const uint4 *p = reinterpret_cast<const uint4 *>(row.in) + first;
            const int fit = whole_fit(first, end);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                if (j * step < fit)
                    Elem<T>::unpack(p[j * step], x[j]);
                else
                    set_empty(j);
            }
        } else {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int64_t v = first + j * step;
                if (v < end)
                    row.load(v, x[j]);
                else
                    set_empty(j);
            }
        }
    }
    // Replace x by e = 2^(x k - s_t) with the tile's own max m_t and
    // s_t = fl(m_t k); return the state (s_t, l_t).  k = log2 e, or
    // scale * log2 e for scaled scores (scale > 0, so the max of x is the max
    // of x * scale).
    // Only the first `live` vectors hold data (the others are empty: -inf);
    // their exponentials are skipped, and values() of them is never asked for.
    __device__ __forceinline__ float2 stats(float k = kLog2e, int live = VPT) {
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < VPT; ++j)
            if (j < live)
#pragma unroll
                for (int i = 0; i < V; ++i) m = fmaxf(m, x[j][i]);
        const float s = m * k;  // -inf stays -inf, +inf stays +inf
        const float shift = safe_shift(s);
        float l = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            if (j >= live) continue;
            float lj = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                x[j][i] = ex2(fmaf(x[j][i], k, -shift));
                lj += x[j][i];
            }
            l += lj;
        }
        return make_float2(s, l);
    }
    __device__ __forceinline__ void values(int j, float f, float *y) const {
#pragma unroll
        for (int i = 0; i < V; ++i) y[i] = x[j][i] * f;
    }
    __device__ __forceinline__ void values_shift(int j, float shift, float f, float *y, float k = kLog2e) const {
#pragma unroll
        for (int i = 0; i < V; ++i) y[i] = ex2(fmaf(x[j][i], k, -shift)) * f;
    }
    // y = e * f (after stats())
    template <bool WHOLE = false>
    __device__ __forceinline__ void scale_store(const RowView<T> &row, int64_t first, int64_t step, int64_t end,
                                                float f) const {
        tile_store<T, VPT, WHOLE>(row, first, step, end, [&](int j, float *y) { values(j, f, y); });
    }
    // y = 2^(x k - shift) * f (the tile as loaded, without stats())
    template <bool WHOLE = false>
    __device__ __forceinline__ void shift_store(const RowView<T> &row, int64_t first, int64_t step, int64_t end,
                                                float shift, float f, float k = kLog2e) const {
        tile_store<T, VPT, WHOLE>(row, first, step, end,
                                  [&](int j, float *y) { values_shift(j, shift, f, y, k); });
    }
};

template <typename T, int VPT>
struct PackedTile {
    static_assert(sizeof(T) == 2, "packed tiles hold 16-bit data");
    static constexpr int V = Elem<T>::kVec;
    uint4 raw[VPT];  // the inputs; after stats(), their exponentials as fp16 pairs

    __device__ __forceinline__ void set(int j, const uint4 &r) { raw[j] = r; }
    __device__ __forceinline__ void load_one(int j, const RowView<T> &row, int64_t v) { raw[j] = row.load_raw(v); }
    __device__ __forceinline__ void set_empty(int j) {
        const uint32_t w = (uint32_t)Elem<T>::kNegInfBits * 0x10001u;
        raw[j] = make_uint4(w, w, w, w);
    }
    template <bool WHOLE = false>
    __device__ __forceinline__ void load(const RowView<T> &row, int64_t first, int64_t step, int64_t end) {
        if constexpr (WHOLE) {
            const uint4 *p = reinterpret_cast<const uint4 *>(row.in) + first;
            const int fit = whole_fit(first, end);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                if (j * step < fit)
                    raw[j] = p[j * step];
                else
                    set_empty(j);
            }
        } else {
            // every vector as an aligned 16-byte load at a constant offset
            // (RowView::vec_in), then the elements of the row's partial end
            // vectors that lie outside the row set to -inf
            const uint4 *p = row.vec_in() + first;
            const int fit = whole_fit(first, end);
            const uint32_t ninf = Elem<T>::kNegInfBits;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                if (j * step < fit)
                    raw[j] = p[j * step];
                else
                    set_empty(j);
            }
            if (first == 0 && row.head != 0 && fit > 0) raw[0] = keep_range16(raw[0], row.head, V, ninf);
            if (row.tail < V) {
                const int64_t last = row.nvec - 1 - first;
#pragma unroll
                for (int j = 0; j < VPT; ++j)
                    if ((int64_t)j * step == last && j * step < fit) raw[j] = keep_range16(raw[j], 0, row.tail, ninf);
            }
        }
    }
    // As FloatTile::stats: only the first `live` vectors hold data.  The
    // exponentials e = 2^(x k - shift), in [0, 1], then replace the inputs in
    // the tile, rounded to fp16 pairs (relative error 2^-11 whatever T is):
    // a result is e * f, one multiply, instead of a second exponential.  With
    // the output rounded once more, |error| <= 2^-11 y + half an ulp of y,
    // inside the 16-bit tolerances (fp16 1e-3, bf16 4e-3).  After stats() the
    // tile holds exponentials, not inputs: shift_store() needs a fresh load.
    __device__ __forceinline__ float2 stats(float k = kLog2e, int live = VPT) {
        // the max on the packed pairs (a NaN never wins, as with fmaxf)
        uint32_t mw = (uint32_t)Elem<T>::kNegInfBits * 0x10001u;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            if (j >= live) continue;
            mw = Elem<T>::max2(mw, raw[j].x);
            mw = Elem<T>::max2(mw, raw[j].y);
            mw = Elem<T>::max2(mw, raw[j].z);
            mw = Elem<T>::max2(mw, raw[j].w);
        }
        const float2 mp = Elem<T>::pair(mw);
        const float m = fmaxf(mp.x, mp.y);
        const float s = m * k;
        const float shift = safe_shift(s);
        float l = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            if (j >= live) {
                raw[j] = make_uint4(0u, 0u, 0u, 0u);
                continue;
            }
            float x[V];
            Elem<T>::unpack(raw[j], x);
            float lj = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                x[i] = ex2(fmaf(x[i], k, -shift));
                lj += x[i];
            }
            l += lj;
            raw[j] = Elem<__half>::pack(x);
        }
        return make_float2(s, l);
    }
    __device__ __forceinline__ void values_shift(int j, float sh, float f, float *y, float k = kLog2e) const {
        float x[V];
        Elem<T>::unpack(raw[j], x);
#pragma unroll
        for (int i = 0; i < V; ++i) y[i] = ex2(fmaf(x[i], k, -sh)) * f;
    }
    // y = e * f from the exponentials stats() left in the tile
    __device__ __forceinline__ void values(int j, float f, float *y) const {
        Elem<__half>::unpack(raw[j], y);
#pragma unroll
        for (int i = 0; i < V; ++i) y[i] *= f;
    }
    // y = e * f (after stats())
    template <bool WHOLE = false>
    __device__ __forceinline__ void scale_store(const RowView<T> &row, int64_t first, int64_t step, int64_t end,
                                                float f) const {
        tile_store<T, VPT, WHOLE>(row, first, step, end, [&](int j, float *y) { values(j, f, y); });
    }
    // y = 2^(x k - shift) * f (the tile as loaded, without stats())
    template <bool WHOLE = false>
    __device__ __forceinline__ void shift_store(const RowView<T> &row, int64_t first, int64_t step, int64_t end,
                                                float shift, float f, float k = kLog2e) const {
        tile_store<T, VPT, WHOLE>(row, first, step, end,
                                  [&](int j, float *y) { values_shift(j, shift, f, y, k); });
    }
};

// fp32 rows keep their exponentials; 16-bit rows stay packed.
template <typename T, int VPT> struct TileSel { using type = PackedTile<T, VPT>; };
template <int VPT> struct TileSel<float, VPT> { using type = FloatTile<float, VPT>; };
template <typename T, int VPT> using Tile = typename TileSel<T, VPT>::type;

}  // namespace mbrs
