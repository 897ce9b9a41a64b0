// tcgen05 (5th-generation tensor core) building blocks for sm_100-family GPUs,
// written from the PTX ISA: shared-memory matrix descriptors, the instruction
// descriptors of kind::f16, TMEM allocation, the tcgen05 fences, commit to an
// mbarrier and TMEM loads (the grouped GEMM issues its MMAs with A in TMEM).
//
// Operand layout used everywhere here: K-major tiles with the 128-byte
// swizzle. A tile of R rows x 64 bf16 columns occupies R * 128 bytes; row r
// starts at 128 r, and its 16-byte chunk c (columns 8c .. 8c+7) is stored at
// chunk position c ^ (r % 8). Tiles start on a 1024-byte boundary (8 rows);
// the stride between 8-row groups is 1024 bytes. An MMA consumes 16 columns
// (32 bytes) of K; stepping K inside the 64-column tile advances the
// descriptor's start address by 32 bytes (the swizzle is a function of the
// address bits, so the step needs no re-layout).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ds4 {
namespace umma {

// Shared-memory matrix descriptor (64 bits):
//   [0,14)  start address >> 4      [16,30) leading-dimension byte offset >> 4
//   [32,46) stride-dimension byte offset >> 4   [46,48) version = 1
//   [49,52) base offset = 0         [61,64) layout: 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t desc_sw128(uint32_t smem_addr) {
    return (uint64_t)((smem_addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B, fp32
// accumulation, both operands K-major, shape M x N:
//   [4,6) D format = 1 (f32)   [7,10) A format = 1 (bf16)   [10,13) B format = 1
//   [15] A major = 0 (K)   [16] B major = 0 (K)   [17,23) N >> 3   [24,29) M >> 4
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The same with binary16 A and B (A format = B format = 0).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Warp-wide: allocate ncols TMEM columns (power of two >= 32); the base
// address is written to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Warp-wide.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// One thread: the mbarrier gets one arrival when all MMAs issued so far by
// this thread have completed.
__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// Warp-wide: 32 lanes x 8 columns of 32-bit TMEM starting at taddr (lane
// field = the warp's lane quarter base). Thread i receives lane base + i.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

} // namespace umma
} // namespace ds4
