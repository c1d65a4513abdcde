/*
 * synth_core.h - the Philox4x32-10 block and the Irwin-Hall deviate, shared by the
 * host (synth.c) and device (synth.cu) fills of this module only.
 * Round constants and key increments are the published Philox4x32 ones
 * (Salmon et al., SC 2011).
 */
#ifndef PP_SYNTH_CORE_H
#define PP_SYNTH_CORE_H
#include <stdint.h>

#ifdef __CUDACC__
#define SYN_FN static __host__ __device__ __forceinline__
#else
#define SYN_FN static inline
#endif

SYN_FN void syn_philox(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                       uint32_t k0, uint32_t k1, uint32_t out[4]) {
  for (int r = 0; r < 10; ++r) {
    uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Centred 8-term Irwin-Hall integer for element idx of (seed, stream). */
SYN_FN int32_t syn_ih8(uint64_t idx, uint32_t seed, uint32_t stream) {
  uint32_t w[4];
  syn_philox((uint32_t)idx, (uint32_t)(idx >> 32), stream, 0u, seed, 0u, w);
  int32_t s = 0;
  for (int j = 0; j < 4; ++j) s += (int32_t)(w[j] & 0xFFFFu) + (int32_t)(w[j] >> 16);
  return s - 262140;
}

SYN_FN uint16_t syn_f32_to_bf16_rne(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t u = v.u;
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)0x7FC0u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

#endif
