// attention.cuh -- fifth-generation tensor-core (tcgen05) building blocks for
// the fused attention forward: tensor-memory allocation, loads and stores,
// shared-memory matrix descriptors, the instruction descriptor, MMA issue and
// completion tracking, and tiled TMA loads.  All of it is inline PTX for
// sm_103a.
#pragma once

#include <cuda.h>  // CUtensorMap (the 128-byte TMA descriptor)
#include <stdint.h>

#include "common.cuh"

namespace mbrs {
namespace attn {

// ---------------------------------------------------------------------------
// Tensor memory (TMEM): 128 lanes x 512 columns of 32-bit cells per SM.  An
// address is (lane << 16) | column.  A warp may touch only the 32 lanes of its
// quarter: warp w of a block reaches lanes 32 (w mod 4) .. 32 (w mod 4) + 31.
// ---------------------------------------------------------------------------
// Whole-warp calls.  alloc writes the base address of `cols` columns (a power
// of two >= 32) into the shared-memory word at slot.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(cols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
// Ordering of tcgen05 operations across a thread synchronisation (a barrier
// or an mbarrier wait): `before` on the side that signals, `after` on the side
// that waits.
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive columns of this thread's lane (shape 32x32b: thread i of the
// warp reads lane base + i) into v[0..31], the load's destination registers
// themselves.  Completes at tmem_wait_ld(); tmem_fence_regs<32>(v) after the
// wait keeps every use of v after it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]),
          "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15]),
          "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]),
          "=f"(v[24]), "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// After tmem_wait_ld(): v[0..N) -- registers a tcgen05.ld filled -- pass
// through empty volatile statements that the compiler must treat as writing
// them.  A load's outputs look ready to the compiler at the load itself, so
// without this it may place arithmetic on them (or copies of them) before the
// wait, reading registers the load has not filled yet.
template <int N>
__device__ __forceinline__ void tmem_fence_regs(float *v) {
    static_assert(N % 8 == 0, "whole groups of eight registers");
#pragma unroll
    for (int i = 0; i < N; i += 8) {
        float *w = v + i;
        asm volatile("" : "+f"(w[0]), "+f"(w[1]), "+f"(w[2]), "+f"(w[3]), "+f"(w[4]), "+f"(w[5]), "+f"(w[6]), "+f"(w[7]));
    }
}

// v[0..31] into 32 consecutive columns of this thread's lane.  Completes at
// tmem_wait_st().
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
// v[0..15] into 16 consecutive columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
    uint32_t u[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(v[i]);
    tmem_st32(taddr, u);
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor (64 bits) for operands in the 128-byte
// swizzled layout: rows of 128 bytes, the 16-byte chunks of row r stored at
// chunk position (chunk XOR (r mod 8)), eight rows (1024 bytes) per swizzle
// atom, atoms 1024-byte aligned -- the layout a TMA load with 128-byte
// swizzle writes.
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-48  0b001 (descriptor version of this architecture)
//   bits 49-51  base offset (0: atoms are 1024-byte aligned)
//   bit  52     leading offset mode (0: relative)
//   bits 61-63  swizzle mode (2: 128-byte)
// K-major operand (K contiguous within a row): the stride offset is the
// distance between 8-row groups (1024 bytes); the leading offset is unused by
// this swizzle and set to 16 bytes.  MN-major operand (M or N contiguous): the
// leading offset is the distance between successive 64-element column blocks,
// the stride offset that between 8-row groups along K.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lead_bytes, uint32_t stride_bytes) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lead_bytes >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((stride_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor (32 bits) of kind::f16 with an fp32 accumulator:
//   bits 4-5 D type (1: f32); bits 7-9 / 10-12 A / B type (0: f16, 1: bf16);
//   bit 15 / 16 A / B major (0: K-major, 1: MN-major); bits 17-22 N >> 3;
//   bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t f16_idesc(bool bf16, bool b_mn_major, int m, int n) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D[tmem] (+)= A[smem] . B[smem]; issued by one thread.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] . B[smem]: A (M x K) held in tensor memory, row m in
// lane m, two 16-bit elements per 32-bit column (element k in the low half
// of column k / 2 when k is even); issued by one thread.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// One arrival on the mbarrier at `bar` once every MMA this thread issued so
// far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Tiled 3-D TMA load (coordinates innermost first) into shared memory,
// completing `bar`'s transaction count.  x * element size must be a multiple
// of 16 bytes; out-of-range elements read as zero.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
        "%4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
// Pairs of fp32 values in one 64-bit register (this architecture's packed
// fp32 arithmetic: one instruction for two round-to-nearest operations).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 f2_split(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// the largest of three (a NaN operand is ignored, as with fmaxf)
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Tiled 3-D TMA store (coordinates innermost first) from shared memory, in
// the thread's bulk async-group; elements outside the tensor are not written.
// x * element size must be a multiple of 16 bytes and no coordinate negative.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int32_t x, int32_t y, int32_t z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the thread's committed bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// the thread's committed bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// order this thread's shared-memory writes before later async-proxy (TMA) reads
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4 &v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace attn
}  // namespace mbrs
