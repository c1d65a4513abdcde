// pp_tcgen05.cuh - 5th-generation tensor-core helpers (sm_103a): shared-memory matrix
// descriptors, instruction descriptors, MMA issue and commit, tensor-memory loads.
#pragma once
#include <stdint.h>

namespace pp {

// Shared-memory matrix descriptor: K-major tile, 128-byte swizzle, 8-row atoms of
// 1024 bytes stacked along M/N (stride 1024), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)(1024u >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: bf16 A and B (K-major), fp32 accumulator.
__host__ __device__ constexpr uint32_t instr_desc(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 8 consecutive accumulator columns of this thread's TMEM lane (no wait).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t r[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Orders a register after the preceding tcgen05.wait::ld (volatile asms keep their order).
__device__ __forceinline__ float after_wait(uint32_t r) {
  asm volatile("" : "+r"(r));
  return __uint_as_float(r);
}

// 2 consecutive accumulator columns of this thread's TMEM lane (no wait).
__device__ __forceinline__ void tmem_ld2(uint32_t taddr, uint32_t r[2]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(taddr));
}

// Shared-memory matrix descriptor, MN-major tile with the 128-byte swizzle: 8 k-rows of
// 128 bytes (64 bf16 along M/N) per 1024-byte atom; atoms follow each other along K
// every 1024 bytes (stride offset) and along M/N every `lbo` bytes (leading offset).
__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t addr, uint32_t lbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)(1024u >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

}  // namespace pp
