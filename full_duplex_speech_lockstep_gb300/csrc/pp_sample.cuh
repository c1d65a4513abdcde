// pp_sample.cuh - the sampling variants of the per-row token decision, one CTA per row.
//
// The pages decode greedily and name the knobs a deployment may turn instead
// (temperature, nucleus top-p, repetition penalty, a separate audio temperature:
// "PersonaPlex ... vLLM-Omni", deployment config; the persona-tuning article,
// generation parameters and repetition penalty).  Taken in this order:
//   1. repetition penalty on the raw logits, the signed form of Keskar et al. (CTRL,
//      2019): each distinct history token's logit is divided by R when positive and
//      multiplied by R otherwise;
//   2. division by the temperature;
//   3. top-k: keep the finite values at or above the k-th largest (ties kept);
//   4. e_i = expf(v_i - max v) over the kept values;
//   5. nucleus: keep e at or above the largest e value whose own mass plus the mass of
//      every larger e reaches p * sum(e) (ties kept);
//   6. inverse CDF in index order: the first kept index whose running mass exceeds
//      u * (kept mass), else the last kept index.
// Values that are not finite are never chosen; with none left the token is 0.
//
// Everything is deterministic: the row sits in shared memory, each threshold is found
// by a 32-step binary search on an order-preserving key with fixed-order block
// reductions, and the running mass is a fixed-order block scan over contiguous
// per-thread chunks.  The random draw u comes from Philox4x64-10 (Salmon et al., SC
// 2011) keyed by the session's seed and counted by (position, row / 4).
#pragma once

#include <math.h>
#include <stdint.h>

#include "pp_internal.cuh"

namespace pp {

constexpr int kHist = 256;                  // text-token history ring per slot
constexpr int kSampleSmemMax = 200 * 1024;  // a row of logits held in shared memory

// Per-slot sampling parameters (device copy of pp_sampling).  A temperature <= 0
// keeps that stream greedy.
struct SampleParams {
  float t_temp;
  int32_t t_top_k;
  float t_top_p;
  float penalty;
  int32_t window;
  float a_temp;
  int32_t a_top_k;
  float a_top_p;
  uint32_t seed_lo, seed_hi;
  int32_t pad[2];
};
static_assert(sizeof(SampleParams) == 48, "device layout");

namespace samp {

__device__ __forceinline__ void philox4x64(uint64_t c[4], uint64_t k0, uint64_t k1) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += W0;
      k1 += W1;
    }
    const uint64_t hi0 = __umul64hi(M0, c[0]), lo0 = M0 * c[0];
    const uint64_t hi1 = __umul64hi(M1, c[2]), lo1 = M1 * c[2];
    const uint64_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// u for row `row` (0 text, 1..8 agent audio) at session position pos: top 24 bits of
// word row % 4 of the block at counter (pos, row / 4, 0, 0), key (seed, 0).
__device__ __forceinline__ float uniform(uint64_t seed, int64_t pos, int row) {
  uint64_t c[4] = {(uint64_t)pos, (uint64_t)(row / 4), 0ull, 0ull};
  philox4x64(c, seed, 0ull);
  uint64_t w = c[0];
  if ((row & 3) == 1) w = c[1];
  if ((row & 3) == 2) w = c[2];
  if ((row & 3) == 3) w = c[3];
  return (float)(w >> 40) * (1.0f / 16777216.0f);
}

// Order-preserving key of a float (-0 folded onto +0).
__device__ __forceinline__ uint32_t fkey(float v) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Fixed-order block reductions: per-warp butterfly, warp totals added in warp order.
template <int NT>
__device__ __forceinline__ float sum(float v) {
  __shared__ float sh[NT / 32 + 1];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < NT / 32; ++w) t += sh[w];
    sh[NT / 32] = t;
  }
  __syncthreads();
  const float r = sh[NT / 32];
  __syncthreads();
  return r;
}

template <int NT>
__device__ __forceinline__ int count(int v) {
  __shared__ int sh[NT / 32 + 1];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < NT / 32; ++w) t += sh[w];
    sh[NT / 32] = t;
  }
  __syncthreads();
  const int r = sh[NT / 32];
  __syncthreads();
  return r;
}

template <int NT, bool kMax>
__device__ __forceinline__ int extreme_i(int v) {
  __shared__ int sh[NT / 32 + 1];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const int x = __shfl_xor_sync(0xffffffffu, v, o);
    v = kMax ? max(v, x) : min(v, x);
  }
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = sh[0];
    for (int w = 1; w < NT / 32; ++w) t = kMax ? max(t, sh[w]) : min(t, sh[w]);
    sh[NT / 32] = t;
  }
  __syncthreads();
  const int r = sh[NT / 32];
  __syncthreads();
  return r;
}

template <int NT>
__device__ __forceinline__ float max_f(float v) {
  __shared__ float sh[NT / 32 + 1];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = sh[0];
    for (int w = 1; w < NT / 32; ++w) t = fmaxf(t, sh[w]);
    sh[NT / 32] = t;
  }
  __syncthreads();
  const float r = sh[NT / 32];
  __syncthreads();
  return r;
}

// Exclusive scan of one float per thread in thread order; *total gets the sum.
template <int NT>
__device__ __forceinline__ float scan_excl(float v, float* total) {
  __shared__ float sh[NT / 32 + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float x = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += x;
  }
  float exc = __shfl_up_sync(0xffffffffu, inc, 1);
  if (lane == 0) exc = 0.f;
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (threadIdx.x == 0) {   // warp offsets, in warp order
    float t = 0.f;
    for (int w = 0; w < NT / 32; ++w) {
      const float x = sh[w];
      sh[w] = t;
      t += x;
    }
    sh[NT / 32] = t;
  }
  __syncthreads();
  const float r = sh[warp] + exc;
  *total = sh[NT / 32];
  __syncthreads();
  return r;
}

}  // namespace samp

// One sampled token of the n logits at lg (global), using sv[n] of shared memory.
// hist holds the history ring (hist_pos >= 0: the n_hist entries before position
// hist_pos, at index (p mod kHist)) or a plain array (hist_pos < 0).  NaN logits raise
// PP_S_NAN in *status.  All threads of the block must call it; all get the token.
template <int NT>
__device__ int block_sample(const float* __restrict__ lg, int n, float temperature, int top_k,
                            float top_p, float penalty, const int32_t* __restrict__ hist,
                            int n_hist, int64_t hist_pos, float u, uint32_t* status,
                            float* sv) {
  __shared__ int32_t s_h[kHist];
  const int tid = threadIdx.x;
  int nan = 0;
  for (int i = tid; i < n; i += NT) {
    const float x = lg[i];
    nan |= isnan(x);
    sv[i] = x;
  }
  if (n_hist > kHist) n_hist = kHist;
  for (int j = tid; j < n_hist; j += NT)
    s_h[j] = hist[hist_pos < 0 ? j : (int)((hist_pos - 1 - j) & (kHist - 1))];
  __syncthreads();
  // 1. repetition penalty, once per distinct token (first occurrence applies it)
  if (penalty != 1.f) {
    for (int j = tid; j < n_hist; j += NT) {
      const int h = s_h[j];
      if (h < 0 || h >= n) continue;
      bool seen = false;
      for (int i = 0; i < j; ++i) seen |= (s_h[i] == h);
      if (seen) continue;
      const float x = sv[h];
      sv[h] = x > 0.f ? x / penalty : x * penalty;
    }
    __syncthreads();
  }
  // 2. temperature, and the maximum over finite values
  float m = -INFINITY;
  int nfin = 0;
  for (int i = tid; i < n; i += NT) {
    const float x = sv[i] / temperature;
    sv[i] = x;
    if (isfinite(x)) {
      m = fmaxf(m, x);
      ++nfin;
    }
  }
  m = samp::max_f<NT>(m);
  nfin = samp::count<NT>(nfin);
  if (nan && status) atomicOr(status, PP_S_NAN);
  if (nfin == 0) return 0;
  // 3. top-k: the largest key whose count of finite keys at or above it reaches k
  uint32_t kk = 0u;
  if (top_k > 0 && top_k < nfin) {
    for (int bit = 31; bit >= 0; --bit) {
      const uint32_t cand = kk | (1u << bit);
      int c = 0;
      for (int i = tid; i < n; i += NT) {
        const float x = sv[i];
        c += (isfinite(x) && samp::fkey(x) >= cand);
      }
      if (samp::count<NT>(c) >= top_k) kk = cand;
    }
  }
  // 4. exponentials of the kept values against the maximum (0 marks a dropped value)
  float z = 0.f;
  for (int i = tid; i < n; i += NT) {
    const float x = sv[i];
    const float e = (isfinite(x) && samp::fkey(x) >= kk) ? expf(x - m) : 0.f;
    sv[i] = e;
    z += e;
  }
  const float Z = samp::sum<NT>(z);
  // 5. nucleus: the largest bit pattern t (e >= 0, so bits order like values) whose
  // mass of e with bits >= t reaches p * Z
  uint32_t tb = 0u;
  if (top_p < 1.f) {
    const float P = top_p * Z;
    for (int bit = 30; bit >= 0; --bit) {
      const uint32_t cand = tb | (1u << bit);
      float ms = 0.f;
      for (int i = tid; i < n; i += NT) {
        const float e = sv[i];
        if (__float_as_uint(e) >= cand) ms += e;
      }
      if (samp::sum<NT>(ms) >= P) tb = cand;
    }
  }
  // 6. inverse CDF over contiguous per-thread chunks, in index order
  const int chunk = (n + NT - 1) / NT;
  const int lo = min(n, tid * chunk), hi = min(n, lo + chunk);
  float loc = 0.f;
  int last = -1;
  for (int i = lo; i < hi; ++i) {
    const float e = sv[i];
    if (e > 0.f && __float_as_uint(e) >= tb) {
      loc += e;
      last = i;
    }
  }
  float total;
  const float excl = samp::scan_excl<NT>(loc, &total);
  const float target = u * total;
  int pick = 0x7FFFFFFF;
  float acc = 0.f;
  for (int i = lo; i < hi; ++i) {
    const float e = sv[i];
    if (!(e > 0.f && __float_as_uint(e) >= tb)) continue;
    acc += e;
    if (excl + acc > target) {
      pick = i;
      break;
    }
  }
  pick = samp::extreme_i<NT, false>(pick);
  if (pick == 0x7FFFFFFF) pick = samp::extreme_i<NT, true>(last);
  return pick < 0 ? 0 : pick;
}

}  // namespace pp
