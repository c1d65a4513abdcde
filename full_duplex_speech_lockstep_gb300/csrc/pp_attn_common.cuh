// pp_attn_common.cuh - work units, error flagging and the final chunk merge shared by
// the two ring-attention kernels (CUDA cores and tensor cores).
#pragma once
#include <math.h>

#include "pp_internal.cuh"

namespace pp {
namespace attn {

struct Unit {
  int s, h, c, nk;   // slot, head, chunk, keys in this chunk (0: skip)
};

__device__ __forceinline__ Unit decode_unit(const AttnArgs& a, int u) {
  Unit r;
  const int pair = u / a.nc_max;
  r.c = u - pair * a.nc_max;
  r.s = pair / a.H;
  r.h = pair - r.s * a.H;
  const int n = min(__ldg(a.n_valid + r.s), a.W);   // never past the W ring positions
  r.nk = min(kAttnChunk, n - r.c * kAttnChunk);
  if (r.nk < 0) r.nk = 0;
  return r;
}

// SMs of the current device (looked up once per device).
inline int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

__device__ __forceinline__ void raise_timeout(const AttnArgs& a, volatile int* s_abort) {
  *s_abort = 1;
  if (a.status) atomicOr(a.status, PP_S_TIMEOUT);
}

// DPL consecutive floats from L2 (4*DPL-byte aligned)
template <int DPL>
__device__ __forceinline__ void ldcg_vec(const float* p, float f[DPL]) {
  if constexpr (DPL == 4) {
    const float4 x = __ldcg(reinterpret_cast<const float4*>(p));
    f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
  } else if constexpr (DPL == 2) {
    const float2 x = __ldcg(reinterpret_cast<const float2*>(p));
    f[0] = x.x; f[1] = x.y;
  } else {
    f[0] = __ldcg(p);
  }
}

// Final merge of one (slot, head) by one warp: the chunk partials in chunk order,
// out = (sum_c f_c o_c) / (sum_c f_c l_c) with f_c = 2^(m_c - max m).  The block's L2
// lines are then discarded: the partials are dead and need never reach HBM.
template <int DH>
__device__ __forceinline__ void merge_pair(const AttnArgs& a, float* part, int nc, int s, int h,
                                           int lane) {
  constexpr int DPL = DH / 32;
  constexpr int R = attn_rec_floats(DH);
  float M = -INFINITY;
  for (int c = lane; c < nc; c += 32) M = fmaxf(M, __ldcg(part + (size_t)c * R));
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f, O[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) O[i] = 0.f;
  for (int c0 = 0; c0 < nc; c0 += 8) {
    float mv[8], lv[8], ov[8][DPL];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int c = c0 + e < nc ? c0 + e : nc - 1;   // clamped reads, masked below
      const float* src = part + (size_t)c * R;
      mv[e] = __ldcg(src);
      lv[e] = __ldcg(src + 1);
      ldcg_vec<DPL>(src + 8 + lane * DPL, ov[e]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (c0 + e < nc) {
        const float f = exp2f(mv[e] - M);
        L = fmaf(f, lv[e], L);
#pragma unroll
        for (int i = 0; i < DPL; ++i) O[i] = fmaf(f, ov[e][i], O[i]);
      }
    }
  }
  const int HD = a.H * DH;
#pragma unroll
  for (int i = 0; i < DPL; ++i) {
    const int col = h * DH + lane * DPL + i;
    const float r = O[i] / L;
    a.out[(size_t)s * a.out_ld + col] = r;
    if (a.op) op_store(a.op, HD, a.op_Bp, s, col, r);
  }
  __syncwarp();
  const int lines = (int)(attn_pair_floats(a.nc_max, DH) * sizeof(float) / 128);
  for (int ln = lane; ln < lines; ln += 32)
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(part + (size_t)ln * 32) : "memory");
}

}  // namespace attn
}  // namespace pp
