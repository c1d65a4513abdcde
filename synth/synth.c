/* synth.c - host fills of the seeded input generator (see synth.h). */
#include "synth.h"
#include "synth_core.h"
#include <math.h>

void ppsyn_philox(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  syn_philox(ctr[0], ctr[1], ctr[2], ctr[3], key[0], key[1], out);
}

float ppsyn_normal_scale(double sigma) {
  /* variance of one 16-bit uniform is (65536^2 - 1) / 12; eight of them are summed */
  double sd = sqrt(8.0 * (65536.0 * 65536.0 - 1.0) / 12.0);
  return (float)(sigma / sd);
}

void ppsyn_normal_bf16_host(uint16_t* out, int64_t n, int64_t i0, uint32_t seed,
                            uint32_t stream, float scale) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float x = (float)syn_ih8((uint64_t)(i0 + i), seed, stream) * scale;
    out[i] = syn_f32_to_bf16_rne(x);
  }
}

void ppsyn_normal_f32_host(float* out, int64_t n, int64_t i0, uint32_t seed,
                           uint32_t stream, float scale) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = (float)syn_ih8((uint64_t)(i0 + i), seed, stream) * scale;
}

void ppsyn_uniform_i32_host(int32_t* out, int64_t n, int64_t i0, uint32_t seed,
                            uint32_t stream, int32_t lo, int32_t hi) {
  uint64_t range = (uint64_t)((int64_t)hi - (int64_t)lo);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint32_t w[4];
    uint64_t idx = (uint64_t)(i0 + i);
    syn_philox((uint32_t)idx, (uint32_t)(idx >> 32), stream, 0u, seed, 0u, w);
    out[i] = lo + (int32_t)(((uint64_t)w[0] * range) >> 32);
  }
}
