// pp_async.cuh - shared-memory mbarriers and bulk asynchronous copies (sm_103a), used
// by the tensor-core contraction and the ring attention.  Every wait is bounded.
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace pp {

constexpr uint32_t kWaitLimit = 1u << 24;   // polls before a wait gives up (default)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred P1;\n mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n"
      " selp.b32 %0, 1, 0, P1;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test: true when the phase with this parity has completed.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred P1;\n mbarrier.test_wait.parity.shared::cta.b64 P1, [%1], %2;\n"
      " selp.b32 %0, 1, 0, P1;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Fault-test word of an engine (pp_test_faults): [0] poll budget of a bounded wait
// (<= 0: kWaitLimit), [1] copies a producer still has to withhold, [2] the kernel
// families that withhold (PP_TEST_*).  A null pointer means the defaults.
constexpr uint32_t kWaitFastPolls = 1024;   // polls before a wait reads its budget

// Poll budget of a bounded wait; the word is read only by a wait that has already
// lasted kWaitFastPolls polls, so a wait that succeeds quickly never loads it.
__device__ __forceinline__ uint32_t wait_budget(const int32_t* test_ctl) {
  if (!test_ctl) return kWaitLimit;
  const int32_t v = *reinterpret_cast<const volatile int32_t*>(test_ctl);
  return v > 0 ? (uint32_t)v : kWaitLimit;
}

// Bounded wait: true when the phase completed, false after the poll budget.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const int32_t* test_ctl = nullptr) {
  for (uint32_t i = 0; i < kWaitFastPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint32_t budget = wait_budget(test_ctl);
  for (uint32_t i = kWaitFastPolls; i < budget; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// True (once, for one producer) when a test asked this kernel family to withhold one
// copy: `armed` is the word's [1] as read at kernel start (> 0: a copy is requested).
__device__ __forceinline__ bool take_withhold(const int32_t* test_ctl, int32_t armed,
                                              int32_t kinds, int32_t family) {
  if (!test_ctl || armed <= 0 || !(kinds & family)) return false;
  return atomicSub(const_cast<int32_t*>(test_ctl) + 1, 1) > 0;
}

// The word's [1] and [2], read at kernel start (zeros without a word).
__device__ __forceinline__ void read_withhold(const int32_t* test_ctl, int32_t& armed,
                                              int32_t& kinds) {
  armed = 0;
  kinds = 0;
  if (test_ctl) {
    armed = reinterpret_cast<const volatile int32_t*>(test_ctl)[1];
    kinds = reinterpret_cast<const volatile int32_t*>(test_ctl)[2];
  }
}

// Contiguous global -> shared copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) that completes `bytes` of the barrier's transaction count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// 2D tiled tensor copy global -> shared through a tensor map.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// 4D tiled tensor copy global -> shared through a tensor map.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// Barrier among `count` threads (a multiple of 32) of the CTA under id 1..15.
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace pp
