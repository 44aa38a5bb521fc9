// tcgen05 (fifth-generation tensor core) helpers for sm_103a: tensor-memory allocation, the MMA of
// kind::f16 with binary32 accumulators in tensor memory (A from shared or tensor memory), commit to an
// mbarrier, stores of registers into tensor memory and loads of the accumulator back into registers;
// shared-memory matrix descriptors for the K-major layout with the 128-byte swizzle (the layout a TMA
// tiled load with CU_TENSOR_MAP_SWIZZLE_128B writes).
//
// K-major, 128-byte swizzle: a tile of R rows x 64 binary16 elements (128 bytes per row) sits at a
// 1024-byte-aligned address; row r occupies bytes r * 128 .. r * 128 + 127, and its 16-byte chunk c
// (elements 8c .. 8c + 7) is stored at chunk position c ^ (r % 8). Groups of 8 rows are 1024 bytes
// apart (the descriptor's stride byte offset). One MMA consumes K = 16 elements (32 bytes of each
// row); the next 16 start 32 bytes further into the same rows.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fpx {

// Shared-memory matrix descriptor: start address >> 4 (bits 0-13), leading byte offset >> 4 (bits
// 16-29; not used by swizzled K-major layouts, set to 16 bytes), stride byte offset >> 4 (bits 32-45:
// 1024 bytes between 8-row groups), the fixed value 1 at bits 46-47, base offset 0 (the tile is
// 1024-byte aligned), swizzle mode 2 = 128-byte swizzle (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
    return (uint64_t)((smem_addr >> 4) & 0x3FFFu) | ((uint64_t)1u << 16) | ((uint64_t)(1024u >> 4) << 32) |
           ((uint64_t)1u << 46) | ((uint64_t)2u << 61);
}

// Instruction descriptor of kind::f16: binary32 accumulator (bits 4-5 = 1), A and B binary16 (bits
// 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N / 8 at bits 17-22, M / 16 at bits 24-28.
__host__ __device__ constexpr uint32_t f16_idesc(uint32_t M, uint32_t N) {
    return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Whole warp: allocates `ncols` tensor-memory columns (a power of two >= 32) and writes their base
// address to the shared word at smem_dst.
__device__ __forceinline__ void tmem_alloc(uint32_t smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_dst), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
// Whole warp (the one that allocated): frees the columns.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// One thread: D[tmem] (+)= A[smem] * B[smem]^T for one M x N x 16 step; accumulate != 0 adds to D.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One thread: D[tmem] (+)= A[tmem] * B[smem]^T for one 128 x N x 16 step with A in tensor memory: row m
// of A in lane m, binary16 elements 2c and 2c + 1 of the K step in column a_tmem + c (low, high half).
__device__ __forceinline__ void tc_mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Whole warp: thread i writes r[0..31] to 32 consecutive columns of tensor-memory lane 32 q + i (q = the
// warp's lane quarter, warp % 4), starting at column col of taddr. tmem_st_wait() makes them complete.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// One thread: the mbarrier at smem address `bar` receives one arrival when every tcgen05.mma this
// thread issued before has completed (their shared-memory reads included).
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Whole warp: 16 consecutive binary32 columns of the warp's 32 tensor-memory lanes (lane quarter
// warp % 4 of the CTA's 128 lanes), starting at column col of taddr: thread i receives lane 32 q + i.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

}  // namespace fpx
