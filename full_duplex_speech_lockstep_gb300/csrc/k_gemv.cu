// k_gemv.cu - CUDA-core weight contraction Y[b, m] (op)= sum_k W[m, k] X[b, k] for every
// slot b, bf16 weights streamed once with 16-byte loads, fp32 activations and
// accumulation, with the epilogue fused: store, residual add, SiLU gating of paired
// gate/up rows, or the depformer's token-embedding add.
//
// Each warp owns one output row (two for SiLU: gate row m and up row M + m); lane l
// accumulates k in {8l .. 8l+7} + 256 j in order, then a fixed butterfly sums the
// lanes.  The arithmetic of column b does not depend on how many slots the engine
// holds, so a session's bits do not depend on its neighbours.
#include <math.h>

#include "pp_internal.cuh"

namespace pp {

namespace {

__device__ __forceinline__ uint4 ld_stream(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void unpack8(const uint4 v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <int NB, int EPI>
__global__ void __launch_bounds__(256) k_gemv(Dims D, GemvArgs a) {
  pdl_wait_and_trigger();
  constexpr int R = (EPI == EPI_SILU) ? 2 : 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x * 8 + warp;
  if (m >= a.M) return;
  const int B = D.B;
  float acc[R][NB];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[r][b] = 0.f;

  const uint16_t* wrow[R];
  wrow[0] = a.W + (size_t)m * a.K;
  if (R == 2) wrow[R - 1] = a.W + (size_t)(m + a.M) * a.K;

  for (int k = lane * 8; k < a.K; k += 256) {
    float w[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) unpack8(ld_stream(wrow[r] + k), w[r]);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (b < B) {
        const float4* xp = reinterpret_cast<const float4*>(a.X + (size_t)b * a.ldx + k);
        const float4 x0 = __ldg(xp), x1 = __ldg(xp + 1);
        const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int t = 0; t < 8; ++t) acc[r][b] = fmaf(w[r][t], xv[t], acc[r][b]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[r][b] += __shfl_xor_sync(0xffffffffu, acc[r][b], o);

#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (b < B && lane == (b & 31)) {
      float* y = a.Y + (size_t)b * a.ldy + m;
      if (EPI == EPI_STORE) {
        *y = acc[0][b];
      } else if (EPI == EPI_ADD) {
        *y += acc[0][b];
      } else if (EPI == EPI_SILU) {
        const float g = acc[0][b], u = acc[R - 1][b];
        *y = g / (1.0f + expf(-g)) * u;
      } else {
        const uint16_t e = a.emb[(size_t)a.tok[b] * a.M + m];
        *y = acc[0][b] + __uint_as_float((uint32_t)e << 16);
      }
    }
  }
}

template <int NB>
cudaError_t gemv_nb(const Dims& D, const GemvArgs& a, cudaStream_t s) {
  const dim3 grid((a.M + 7) / 8);
  switch (a.epi) {
    case EPI_STORE: { cudaError_t e_ = launch_k(k_gemv<NB, EPI_STORE>, dim3(grid), dim3(256), 0, s, 1, D, a); if (e_ != cudaSuccess) return e_; } break;
    case EPI_ADD: { cudaError_t e_ = launch_k(k_gemv<NB, EPI_ADD>, dim3(grid), dim3(256), 0, s, 1, D, a); if (e_ != cudaSuccess) return e_; } break;
    case EPI_SILU: { cudaError_t e_ = launch_k(k_gemv<NB, EPI_SILU>, dim3(grid), dim3(256), 0, s, 1, D, a); if (e_ != cudaSuccess) return e_; } break;
    case EPI_EMB: { cudaError_t e_ = launch_k(k_gemv<NB, EPI_EMB>, dim3(grid), dim3(256), 0, s, 1, D, a); if (e_ != cudaSuccess) return e_; } break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const Dims& D, const GemvArgs& a, cudaStream_t s) {
  if (a.K % 8 != 0) return cudaErrorInvalidValue;
  const int B = D.B;
  if (B <= 1) return gemv_nb<1>(D, a, s);
  if (B <= 2) return gemv_nb<2>(D, a, s);
  if (B <= 4) return gemv_nb<4>(D, a, s);
  if (B <= 8) return gemv_nb<8>(D, a, s);
  if (B <= 16) return gemv_nb<16>(D, a, s);
  if (B <= 32) return gemv_nb<32>(D, a, s);
  return gemv_nb<64>(D, a, s);
}

}  // namespace pp
