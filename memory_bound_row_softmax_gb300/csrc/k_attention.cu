// k_attention.cu -- fused attention forward on the fifth-generation tensor cores:
//
//     O = softmax(Q K^T * sm_scale, causal: key j <= query i) V
//
// for every (batch, head), with Q, K, V, O stored [batch, heads, n_ctx, 128]
// (page "Dissecting Memory Bandwidth & SRAM Tiling in Triton: From GEMM to
// FlashAttention-3", sections "The Mathematical Remedy: Online Softmax
// Tiling" and "Writing the Kernel in OpenAI Triton": tiles of 128 queries,
// running max and normaliser per query, the output accumulator rescaled when
// the max moves, P rounded to the input type before the second product, the
// accumulator divided by the normaliser at the end).
//
// A persistent grid, one block per SM, works through items of 256 queries of
// one head: two query tiles A and B of 128.  320 threads in four roles:
//   warp 8, one lane  -- fetches the next item and publishes it to the block;
//                        TMA: the item's two Q tiles, then K_0, V_0, K_1,
//                        V_1, ... (tiles of 128 keys, 128-byte swizzled rows)
//                        into a ring of kSlots shared-memory slots;
//   warp 9, one lane  -- tcgen05.mma: S_t = Q_t K_j^T into tensor memory (TMEM)
//                        and O_t += P_t V_j, with P_t read from TMEM where the
//                        softmax wrote it over S_t; warp 9 owns the TMEM
//                        allocation;
//   warps 0-3 / 4-7   -- softmax of tile A / B: thread r of the group owns
//                        query row r of its tile, which is TMEM lane r, so the
//                        row max and row sum are thread-local (no shuffles, no
//                        shared-memory reduction); the exponent arguments and
//                        the sums run as packed fp32 pairs.  Each warp makes
//                        one arrival on its group's P barrier per tile.  At
//                        the end of an item the same threads read O from TMEM,
//                        divide by the normaliser and write their rows into a
//                        shared-memory staging tile, which thread 0 of the
//                        group stores with TMA.
// The two softmax groups take turns with the tensor core: while group A turns
// S_A into P_A, the tensor core computes P_B V and the next S_B, and the
// other way round.  Per key tile the MMA thread issues, in this order,
// O_A += P_A V_j, S_A = Q_A K_{j+1}^T, O_B += P_B V_j, S_B = Q_B K_{j+1}^T:
// MMAs from one thread run in order, so S_t of the next tile overwrites P_t
// only after the product that reads it, and by the time S_t of a tile is
// complete the previous O_t update is too (the softmax may rescale O_t then).
// The running max moves lazily: the shift m used for exp only changes when a
// tile's max exceeds it by more than 2^8 (in log2 units), so O in TMEM is
// rescaled rarely; both O and the normaliser carry the same shift, which
// cancels in O / l, and entries of P stay below 2^8.
//
// Every wait is bounded: a wait that runs out sets the device error word and
// an abort flag the other roles see, outstanding TMA loads and MMAs are
// waited for (bounded), TMEM is released and the block returns.
#include <atomic>
#include <mutex>

#include "attention.cuh"
#include "attention_launch.h"
#include "launch.h"

namespace mbrs {
namespace attn {

__device__ unsigned int g_attn_error;

namespace {

constexpr int kBlockM = 128;  // queries per tile (= TMEM lanes)
constexpr int kBlockN = 128;  // keys per tile
constexpr int kHeadDim = kAttnHeadDim;
constexpr int kTiles = 2;     // query tiles per block, one softmax warpgroup each
constexpr int kRowsPerBlock = kTiles * kBlockM;
constexpr int kThreads = 320;  // warps 0-7 softmax, 8 TMA, 9 MMA
constexpr int kWarpTma = 8, kWarpMma = 9;
// K / V ring: load n (K_{n/2} or V_{n/2}) goes to slot n mod kSlots (measured:
// 3 slots run as fast as 5 or faster -- the K/V tiles come from L2)
constexpr int kSlots = 3;
constexpr uint32_t kTileBytes = kBlockN * kHeadDim * 2;  // one 128 x 128 tile of 16-bit elements
constexpr uint32_t kHalfBytes = kTileBytes / 2;          // its 64-column half: 128 rows of 128 bytes
// shared memory, from a 1024-byte aligned base
constexpr uint32_t kOffQ = 0;                        // Q tile t at kOffQ + t kTileBytes
constexpr uint32_t kOffRing = kTiles * kTileBytes;   // slot i at kOffRing + i kTileBytes
constexpr uint32_t kOffO = kOffRing + kSlots * kTileBytes;  // O_t staged for its TMA store at kOffO + t kTileBytes
constexpr uint32_t kOffBar = kOffO + kTiles * kTileBytes;
enum : int {
    kBarQ = 0,
    kBarFull = 1,                 // + slot: the load landed
    kBarEmpty = 1 + kSlots,       // + slot: its last MMA completed
    kBarS = 1 + 2 * kSlots,       // + tile: S_t is in TMEM
    kBarP = kBarS + kTiles,       // + tile: P_t is in TMEM (one arrival per warp of the group)
    kBarO = kBarP + kTiles,       // + tile: O_t is final
    kBarDrain = kBarO + kTiles,
    kBarItem = kBarDrain + 1,    // the next ring entry of items is published
    kBarQEmpty = kBarItem + 1,   // the item's S products are done with Q
    kBarStage = kBarQEmpty + 1,  // + tile: O_t's staging tile is free (its last store has read it)
    kBarStaged = kBarStage + kTiles,  // + tile: O_t is staged (128 arrivals)
    kNumBars = kBarStaged + kTiles
};
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
constexpr uint32_t kOffItems = kOffAbort + 4;      // two-entry ring of item indices
constexpr size_t kSmemBytes = kOffItems + 8 + 1024;  // + slack for aligning the base
// tensor memory: tile t has S_t (P_t over its first 64 columns) at 128 t and
// O_t at 256 + 128 t
constexpr uint32_t kTmemCols = 512;
constexpr float kShiftSlack = 8.f;  // log2 units

__host__ __device__ constexpr uint32_t col_s(int t) { return 128u * (uint32_t)t; }
__host__ __device__ constexpr uint32_t col_o(int t) { return 256u + 128u * (uint32_t)t; }

static_assert(kSmemBytes <= 227 * 1024, "shared memory per block");
static_assert(kBlockM == 128 && kBlockN == 128 && kHeadDim == 128, "tile shapes the descriptors assume");
static_assert(col_o(kTiles - 1) + kHeadDim <= kTmemCols, "tensor memory columns");

template <typename T> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);  // a at the lower address
    return *reinterpret_cast<const uint32_t *>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void flag_timeout(volatile uint32_t *abort_flag) {
    *abort_flag = 1u;
    atomicOr(&g_attn_error, kErrWaitTimeout);
}

// Wait for phase `parity` of the mbarrier at bar; false once the block is
// aborting or after limit_ns (which starts the abort).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                           uint32_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint32_t t0 = global_timer_lo();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_lo() - t0 > limit_ns) break;
    }
    flag_timeout(abort_flag);
    return false;
}
// The same without the abort check: waits for work already in flight (TMA
// loads, MMAs) before the block lets go of its memory.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                            uint32_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return;
    const uint32_t t0 = global_timer_lo();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return;
        if (global_timer_lo() - t0 > limit_ns) break;
    }
    flag_timeout(abort_flag);
}

}  // namespace


// Work items are 256-query blocks of one head.  Item i (in the order the
// blocks are handed out) maps to (head, block) so that heads go in groups of
// `group` heads (sized by the host so that a group's K and V fit in L2 with
// room to spare) and, within a group, the heaviest blocks come first: every
// head's last block (the most keys under a causal mask), then every head's
// second-to-last, and so on.  Resident blocks then share the group's K and V
// in L2, and handing items out in this order to whichever block is free is
// longest-first list scheduling within the group.
struct Item {
    int bh, mb;
};
__device__ __forceinline__ Item decode_item(int i, int m_blocks, int heads_total, int group) {
    const int per_group = group * m_blocks;
    const int grp = i / per_group;
    const int within = i - grp * per_group;
    const int g0 = grp * group;
    const int heads_here = min(group, heads_total - g0);
    return Item{g0 + within % heads_here, m_blocks - 1 - within / heads_here};
}

// Per-launch work counters (next item, finished blocks).  A launch uses the
// caller's two words when it is given them (work_ext), else slot `work_slot`
// of this array (the host cycles through kWorkSlots); the last block to
// finish resets the counters to zero for their next user.
constexpr int kWorkSlots = 64;
__device__ unsigned int g_work[kWorkSlots][2];

// One block per SM, persistent: the TMA lane fetches items from the slot's
// counter and publishes each to the block through a two-entry ring in shared
// memory; every role walks the same items.  Barrier phases run on across
// items: the K/V ring by load count, S and P by tile count, Q and O by item
// count.  The next item's Q is loaded as soon as the current item's last S
// product has completed (kBarQEmpty), so its loads and first S products
// overlap the current item's last PV product and its epilogue.  The first PV
// product of an item overwrites O_t only after the softmax group has read
// the previous item's O_t: the group reads it before it writes the new item's
// first P_t, which that product waits for.
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    k_attention_fwd(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to, int n_ctx,
                    int m_blocks,
                    int heads_total, int group, unsigned int *work_ext, int work_slot, float kscale, int causal,
                    uint32_t wait_ns, int starve) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    volatile uint32_t *const abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + kOffAbort);
    volatile int *const item_ring = reinterpret_cast<volatile int *>(gbase + kOffItems);
    const auto bar = [base](int i) { return base + kOffBar + 8u * (uint32_t)i; };

    const int warp = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31);
    const int total = heads_total * m_blocks;
    const int n_all = (n_ctx + kBlockN - 1) / kBlockN;
    // key tiles of tile A (queries m0 ..) and B (m0 + 128 ..) of block mb: under
    // the causal mask up to each one's diagonal tile, never past the last key
    const auto tiles_a = [=](int mb) { return causal ? min(2 * mb + 1, n_all) : n_all; };
    const auto tiles_b = [=](int mb) { return causal ? min(2 * mb + 2, n_all) : n_all; };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i)
            mbar_init(bar(i), (i == kBarP || i == kBarP + 1) ? kBlockM / 32
                              : (i == kBarStaged || i == kBarStaged + 1) ? kBlockM : 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == kWarpTma && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&to);
    }
    if (warp == kWarpMma) {
        tmem_alloc(base + kOffTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(gbase + kOffTmemSlot);

    if (warp == kWarpTma) {
        // ---- item fetch and TMA producer ----------------------------------
        if (lane == 0) {
            unsigned int *const work = work_ext ? work_ext : g_work[work_slot];
            int n = 0;  // loads issued so far (all items)
            int k = 0;  // items published so far
            bool ok = true;
            for (;; ++k) {
                // the previous item's S products must be done with Q before
                // the next item (or the end mark) is published: by then every
                // role has read the previous entry, so the ring never runs two
                // entries ahead of a reader
                if (k > 0 && ok) ok = wait_phase(bar(kBarQEmpty), (k - 1) & 1, abort_flag, wait_ns);
                const int item = ok ? (int)atomicAdd(&work[0], 1u) : total;
                item_ring[k & 1] = item < total ? item : -1;
                mbar_arrive(bar(kBarItem));  // release: the entry is visible to whoever waits
                if (item >= total) break;
                const Item it = decode_item(item, m_blocks, heads_total, group);
                const int m0 = it.mb * kRowsPerBlock;
                if (!(starve && k == 0)) {  // the test hook leaves the first Q barrier unarmed
                    mbar_arrive_expect_tx(bar(kBarQ), kTiles * kTileBytes);
                    for (int t = 0; t < kTiles; ++t) {
                        const uint32_t dst = base + kOffQ + (uint32_t)t * kTileBytes;
                        tma_load_3d(dst, &tq, 0, m0 + t * kBlockM, it.bh, bar(kBarQ));
                        tma_load_3d(dst + kHalfBytes, &tq, 64, m0 + t * kBlockM, it.bh, bar(kBarQ));
                    }
                }
                const int loads = 2 * tiles_b(it.mb);
                for (int i = 0; i < loads; ++i, ++n) {
                    const int slot = n % kSlots;
                    // the slot last held load n - kSlots; its MMAs must be done
                    if (n >= kSlots &&
                        !(ok = wait_phase(bar(kBarEmpty + slot), ((n / kSlots) - 1) & 1, abort_flag, wait_ns)))
                        break;
                    const uint32_t dst = base + kOffRing + (uint32_t)slot * kTileBytes;
                    const CUtensorMap *map = (i & 1) ? &tv : &tk;
                    const int y = (i >> 1) * kBlockN;
                    mbar_arrive_expect_tx(bar(kBarFull + slot), kTileBytes);
                    tma_load_3d(dst, map, 0, y, it.bh, bar(kBarFull + slot));
                    tma_load_3d(dst + kHalfBytes, map, 64, y, it.bh, bar(kBarFull + slot));
                }
            }
            // every load issued lands before the block may exit: the last Q
            // and the last kSlots ring loads (earlier ones were consumed)
            if (k > 0 && !(starve && k == 1)) drain_phase(bar(kBarQ), (k - 1) & 1, abort_flag, wait_ns);
            for (int nn = (n > kSlots ? n - kSlots : 0); nn < n; ++nn)
                drain_phase(bar(kBarFull + nn % kSlots), (nn / kSlots) & 1, abort_flag, wait_ns);
            // this block takes no more items: the last one to get here resets
            // the launch's counters
            __threadfence();
            if (atomicAdd(&work[1], 1u) == gridDim.x - 1) {
                work[0] = 0u;
                work[1] = 0u;
                __threadfence();
            }
        }
    } else if (warp == kWarpMma) {
        // ---- MMA issuer ----------------------------------------------------
        if (lane == 0) {
            constexpr uint32_t id_s = f16_idesc(kBf16, false, kBlockM, kBlockN);  // S = Q K^T
            constexpr uint32_t id_o = f16_idesc(kBf16, true, kBlockM, kHeadDim);  // O += P V
            int nb = 0;               // first load of the current item
            int p_cnt[kTiles] = {0, 0};  // P tiles consumed so far, per query tile
            const auto landed = [&](int n) {
                return wait_phase(bar(kBarFull + n % kSlots), (n / kSlots) & 1, abort_flag, wait_ns);
            };
            // S_t = Q_t K_j^T (K_j = load nb + 2j): K = head dim, 8 steps of 16;
            // both operands K-major in shared memory
            const auto issue_s = [&](int t, int j) {
                const uint32_t kb = base + kOffRing + (uint32_t)((nb + 2 * j) % kSlots) * kTileBytes;
                const uint32_t qb = base + kOffQ + (uint32_t)t * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * kHalfBytes + (uint32_t)(kk & 3) * 32u;
                    mma_ss(tmem + col_s(t), sw128_desc(qb + off, 16, 1024), sw128_desc(kb + off, 16, 1024), id_s,
                           kk > 0);
                }
                mma_commit(bar(kBarS + t));
            };
            // O_t += P_t V_j (V_j = load nb + 2j + 1): K = keys, 8 steps of 16;
            // P_t in TMEM (16 keys = 8 columns per step), V_j MN-major in
            // shared memory (head dim contiguous, its two 64-column halves
            // kHalfBytes apart)
            const auto issue_pv = [&](int t, int j) {
                const uint32_t vb = base + kOffRing + (uint32_t)((nb + 2 * j + 1) % kSlots) * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    mma_ts(tmem + col_o(t), tmem + col_s(t) + (uint32_t)kk * 8u,
                           sw128_desc(vb + (uint32_t)kk * 16u * 128u, kHalfBytes, 1024), id_o, (j > 0 || kk > 0));
            };
            const auto wait_p = [&](int t) {
                const bool r = wait_phase(bar(kBarP + t), p_cnt[t] & 1, abort_flag, wait_ns);
                ++p_cnt[t];
                return r;
            };
            bool ok = true;
            for (int k = 0; ok; ++k) {
                if (!(ok = wait_phase(bar(kBarItem), k & 1, abort_flag, wait_ns))) break;
                const int item = item_ring[k & 1];
                if (item < 0) break;
                const int mb = decode_item(item, m_blocks, heads_total, group).mb;
                const int n_a = tiles_a(mb), n_b = tiles_b(mb);
                if (!(ok = wait_phase(bar(kBarQ), k & 1, abort_flag, wait_ns) && landed(nb))) break;
                tc_fence_after();
                // S_t of the new item overwrites P_t of the previous one only
                // after the PV product that reads it (issued earlier, in order)
                issue_s(0, 0);
                issue_s(1, 0);
                mma_commit(bar(kBarEmpty + nb % kSlots));  // K_0 done
                for (int j = 0; j < n_b; ++j) {
                    if (!(ok = landed(nb + 2 * j + 1))) break;  // V_j
                    const bool more_a = j + 1 < n_a, more_b = j + 1 < n_b;
                    if (j < n_a) {
                        if (!(ok = wait_p(0))) break;
                        tc_fence_after();
                        issue_pv(0, j);
                        if (more_a) {
                            if (!(ok = landed(nb + 2 * j + 2))) break;  // K_{j+1}
                            tc_fence_after();
                            issue_s(0, j + 1);
                        } else {
                            mma_commit(bar(kBarO + 0));
                        }
                    }
                    if (!(ok = wait_p(1))) break;
                    tc_fence_after();
                    issue_pv(1, j);
                    mma_commit(bar(kBarEmpty + (nb + 2 * j + 1) % kSlots));  // V_j done
                    if (more_b) {
                        if (!more_a && !(ok = landed(nb + 2 * j + 2))) break;  // K_{j+1}, unless waited above
                        tc_fence_after();
                        issue_s(1, j + 1);
                        mma_commit(bar(kBarEmpty + (nb + 2 * j + 2) % kSlots));  // K_{j+1} done
                    } else {
                        mma_commit(bar(kBarO + 1));
                    }
                    // Q is free once the item's last S product is done; it is
                    // signalled no earlier than after both groups' first P of
                    // the item, so that both have read the item's ring entry
                    // before the producer can publish the entry after next
                    if (j + 2 == n_b || (n_b == 1 && j == 0)) mma_commit(bar(kBarQEmpty));
                }
                nb += 2 * n_b;
            }
            // every MMA issued completes before TMEM is released
            mma_commit(bar(kBarDrain));
            drain_phase(bar(kBarDrain), 0, abort_flag, wait_ns);
        }
    } else {
        // ---- softmax: thread r of group t owns query row r of tile t -------
        const int t = warp >> 2;
        const int r = (int)(threadIdx.x & 127);
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        int s_cnt = 0;  // S tiles consumed so far
        bool ok = true;
        for (int k = 0; ok; ++k) {
            ok = __all_sync(0xffffffffu, wait_phase(bar(kBarItem), k & 1, abort_flag, wait_ns));
            if (!ok) break;
            const int item = item_ring[k & 1];
            if (item < 0) break;
            const Item it = decode_item(item, m_blocks, heads_total, group);
            const int q = it.mb * kRowsPerBlock + t * kBlockM + r;
            const int n_t = t ? tiles_b(it.mb) : tiles_a(it.mb);
            const int q_lim = causal ? min(q + 1, n_ctx) : n_ctx;  // keys [0, q_lim) are kept
            float m_run = -INFINITY;  // the shift, in log2 units
            float l_run = 0.f;
            for (int j = 0; j < n_t; ++j) {
                ok = __all_sync(0xffffffffu, wait_phase(bar(kBarS + t), s_cnt & 1, abort_flag, wait_ns));
                ++s_cnt;
                if (!ok) break;
                tc_fence_after();
                float s[kBlockN];
#pragma unroll
                for (int c = 0; c < kBlockN / 32; ++c)
                    tmem_ld32(lane_addr + col_s(t) + c * 32, s + c * 32);
                tmem_wait_ld();
                tmem_fence_regs<kBlockN>(s);
                const int lim = q_lim - j * kBlockN;  // kept columns of this tile: [0, lim)
                if (lim < kBlockN) {
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c)
                        if (c >= lim) s[c] = -INFINITY;
                }
                float mx[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) mx[i] = s[i];
#pragma unroll
                for (int c = 4; c < kBlockN; c += 8) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) mx[i] = max3(mx[i], s[c + i], s[c + 4 + i]);
                }
                const float m_tile = max3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * kscale;
                float alpha = 1.f;
                bool moved = false;
                if (m_tile > m_run + kShiftSlack) {
                    alpha = ex2(m_run - m_tile);  // 0 on the first tile
                    l_run *= alpha;
                    m_run = m_tile;
                    moved = j > 0;
                }
                // p = 2^(s kscale - m_run), rounded to T in pairs and written
                // over S_t's first 64 columns, in quarters of 32 keys (this
                // thread's S values are all in registers already)
                // (the exponent arguments and the sums in packed fp32 pairs)
                const uint64_t k2 = f2(kscale, kscale), nm2 = f2(-m_run, -m_run);
                uint64_t sum2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float2 a = f2_split(fma_f2(f2(s[32 * h + 2 * c], s[32 * h + 2 * c + 1]), k2, nm2));
                        const float p0 = ex2(a.x), p1 = ex2(a.y);
                        sum2[c & 1] = add_f2(sum2[c & 1], f2(p0, p1));
                        pk[c] = pack2<T>(p0, p1);
                    }
                    tmem_st16(lane_addr + col_s(t) + 16 * h, pk);
                }
                const float2 sa = f2_split(sum2[0]), sb = f2_split(sum2[1]);
                l_run += (sa.x + sa.y) + (sb.x + sb.y);
                if (__any_sync(0xffffffffu, moved)) {
                    // O_t += P_t V_{j-1} has completed (S_t of this tile was
                    // issued after it).  The whole warp takes part (TMEM
                    // accesses are warp-wide); rows whose shift did not move
                    // scale by 1.
#pragma unroll
                    for (int c = 0; c < kHeadDim / 32; ++c) {
                        float ov[32];
                        tmem_ld32(lane_addr + col_o(t) + c * 32, ov);
                        tmem_wait_ld();
                        tmem_fence_regs<32>(ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] *= alpha;
                        tmem_st32(lane_addr + col_o(t) + c * 32, ov);
                    }
                }
                // one arrival per warp, once all its lanes' P (and O) stores
                // have completed
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarP + t));
            }
            if (!ok) break;
            ok = __all_sync(0xffffffffu, wait_phase(bar(kBarO + t), k & 1, abort_flag, wait_ns));
            if (!ok) break;
            tc_fence_after();
            // The epilogue: O_t / l into the staging tile (the TMA box layout:
            // two 64-column halves of 128-byte rows, 16-byte chunks swizzled by
            // the row), then one TMA store per half by thread 0 of the group.
            // Thread 0 first lets the group know the previous item's store has
            // read the tile; the group's writes reach the async proxy (fence)
            // before it issues the store.  Rows past n_ctx are not stored.
            const float inv = 1.f / l_run;
            const uint32_t stage = base + kOffO + (uint32_t)t * kTileBytes;
            if (r == 0) {
                bulk_wait_read_all();
                mbar_arrive(bar(kBarStage + t));
            }
            ok = __all_sync(0xffffffffu, wait_phase(bar(kBarStage + t), k & 1, abort_flag, wait_ns));
            if (!ok) break;
#pragma unroll
            for (int c = 0; c < kHeadDim / 32; ++c) {  // 32 columns of O at a time
                float ov[32];
                tmem_ld32(lane_addr + col_o(t) + c * 32, ov);
                tmem_wait_ld();
                tmem_fence_regs<32>(ov);
#pragma unroll
                for (int v = 0; v < 4; ++v) {  // 16-byte chunk 4c + v of the row
                    uint4 w;
                    w.x = pack2<T>(ov[8 * v + 0] * inv, ov[8 * v + 1] * inv);
                    w.y = pack2<T>(ov[8 * v + 2] * inv, ov[8 * v + 3] * inv);
                    w.z = pack2<T>(ov[8 * v + 4] * inv, ov[8 * v + 5] * inv);
                    w.w = pack2<T>(ov[8 * v + 6] * inv, ov[8 * v + 7] * inv);
                    const uint32_t chunk = (uint32_t)(4 * c + v);
                    const uint32_t row = stage + (chunk >> 3) * kHalfBytes + (uint32_t)r * 128u;
                    st_shared_v4(row + (((chunk & 7u) ^ (uint32_t)(r & 7)) << 4), w);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(kBarStaged + t));
            bool staged = true;
            if (r == 0) {
                staged = wait_phase(bar(kBarStaged + t), k & 1, abort_flag, wait_ns);
                if (staged) {
                    const int32_t y = it.mb * kRowsPerBlock + t * kBlockM;
                    tma_store_3d(&to, stage, 0, y, it.bh);
                    tma_store_3d(&to, stage + kHalfBytes, 64, y, it.bh);
                    bulk_commit();
                }
            }
            ok = __all_sync(0xffffffffu, staged);
            if (!ok) break;
            // this group's reads of O_t are done before it writes the next
            // item's first P_t (tcgen05.wait::ld above, fence before the
            // arrival that the next item's first PV product waits for)
        }
        if (r == 0) bulk_wait_all();  // the stores are complete before the block exits
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (the
// library does not link the driver library itself).
EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

// [batch * heads, n_ctx, 128] viewed as a 3-D tensor (head dim innermost);
// boxes of 64 x 128 x 1 elements (128-byte rows) with 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *ptr, int dtype, int64_t n_ctx, int64_t bh) {
    const EncodeTiled enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)n_ctx, (cuuint64_t)bh};
    const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)n_ctx * kHeadDim * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)kBlockN, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, dtype == kAttnBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
               const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;

template <typename T>
cudaError_t go(const AttnArgs &a, int64_t wait_ns, int starve) {
    static std::atomic<unsigned long long> opted{0};
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (device & (kMaxDevices - 1));
    if (!(opted.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(k_attention_fwd<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        opted.fetch_or(bit, std::memory_order_acq_rel);
    }
    const int64_t bh = a.batch * a.heads;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, a.q, a.dtype, a.n_ctx, bh) || !make_map(&mk, a.k, a.dtype, a.n_ctx, bh) ||
        !make_map(&mv, a.v, a.dtype, a.n_ctx, bh) || !make_map(&mo, a.o, a.dtype, a.n_ctx, bh))
        return cudaErrorInvalidValue;
    const int64_t m_blocks = (a.n_ctx + kRowsPerBlock - 1) / kRowsPerBlock;
    const int group = attention_head_group(bh, a.n_ctx);
    const float kscale = a.sm_scale * kLog2e;
    const uint32_t limit = (uint32_t)std::min<int64_t>(std::max<int64_t>(wait_ns, 1), 0x7fffffff);
    // one persistent block per SM (at most one per item); a launch without
    // the caller's counters takes the next slot of the library's
    static std::atomic<unsigned> launches{0};
    const int slot =
        a.counter ? 0 : (int)(launches.fetch_add(1, std::memory_order_relaxed) % kWorkSlots);
    const int64_t grid = std::min<int64_t>(std::max(a.sms, 1), bh * m_blocks);
    k_attention_fwd<T><<<(unsigned)grid, kThreads, kSmemBytes, a.stream>>>(
        mq, mk, mv, mo, (int)a.n_ctx, (int)m_blocks, (int)bh, group, a.counter, slot, kscale,
        a.causal, limit, starve ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnArgs &a, int64_t wait_ns, int starve) {
    return a.dtype == kAttnBf16 ? go<__nv_bfloat16>(a, wait_ns, starve) : go<__half>(a, wait_ns, starve);
}

int attention_head_group(int64_t heads_total, int64_t n_ctx) {
    const int64_t kv_bytes = n_ctx * kHeadDim * 2 * 2;  // one head's K and V
    const int64_t g = kAttnGroupBytes / std::max<int64_t>(kv_bytes, 1);
    return (int)std::max<int64_t>(1, std::min<int64_t>(g, heads_total));
}

int64_t attention_items(int64_t batch, int64_t heads, int64_t n_ctx) {
    return batch * heads * ((n_ctx + kRowsPerBlock - 1) / kRowsPerBlock);
}

size_t attention_smem_bytes() { return kSmemBytes; }
int attention_threads() { return kThreads; }
int attention_tmem_columns() { return (int)kTmemCols; }

cudaError_t read_clear_attn_error_word(unsigned int *word) {
    cudaError_t e = cudaMemcpyFromSymbol(word, g_attn_error, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_attn_error, &zero, sizeof(unsigned int), 0, cudaMemcpyHostToDevice);
}

}  // namespace attn
}  // namespace mbrs
