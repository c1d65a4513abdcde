// k_attn.cu - split-K sliding-window decode attention over each slot's ring KV.
//
// For slot s at position p the valid ring indices are 0 .. n-1 with n = min(p+1, W):
// before the ring wraps they hold positions 0..p in place, after it every index holds
// one of the last W positions.  Softmax is invariant to the order of its keys, so the
// kernel attends over ring indices directly.
//
// Grid (chunk, head, slot); a CTA of 8 warps covers 256 consecutive ring indices
// (32 per warp).  Within a warp, a group of 4 lanes owns one key: each lane holds a
// quarter of the head's 16-byte pieces of q and loads the matching pieces of K and V
// with streaming 16-byte loads.  The warp partials are merged in warp order, then the
// chunk partial (max, sum, unnormalised output) is written; the last CTA of a
// (slot, head) to finish merges the chunks in chunk order.  Every reduction order is
// fixed by ring index alone, so results are independent of other slots and of timing.
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

template <int DH>
__global__ void __launch_bounds__(kAttnWarps * 32, 4) k_attn(AttnArgs a) {
  pdl_wait_and_trigger();
  constexpr int PIECES = DH / 8;        // 16-byte pieces per K/V row
  constexpr int LOADS = PIECES / 4;     // pieces per lane (4 lanes per key)
  constexpr int ITER = 32 / 8;          // 8 keys per warp iteration, 32 keys per warp
  static_assert(PIECES % 4 == 0, "head dim must be a multiple of 32");
  const int c = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, qd = lane & 3;
  const int HD = a.H * DH;
  float* o_out = a.out + (size_t)s * a.out_ld + h * DH;

  const int n = min(a.n_valid[s], a.W);   // never read past the W ring positions
  if (n <= 0) {   // closed slot: zero output
    if (c == 0)
      for (int i = threadIdx.x; i < DH; i += blockDim.x) {
        o_out[i] = 0.f;
        if (a.op) op_store(a.op, HD, a.op_Bp, s, h * DH + i, 0.f);
      }
    return;
  }
  const int nc = (n + kAttnChunk - 1) / kAttnChunk;
  if (c >= nc) return;

  const size_t blk = (size_t)a.W * DH;
  const uint16_t* Kh = a.k + (size_t)s * a.slot_stride + h * blk;
  const uint16_t* Vh = a.v + (size_t)s * a.slot_stride + h * blk;

  float q[LOADS][8];
  const float* qp = a.q + (size_t)s * a.q_ld + h * DH;
#pragma unroll
  for (int j = 0; j < LOADS; ++j) {
    const float4* p4 = reinterpret_cast<const float4*>(qp + (j * 4 + qd) * 8);
    const float4 a0 = p4[0], a1 = p4[1];
    q[j][0] = a0.x; q[j][1] = a0.y; q[j][2] = a0.z; q[j][3] = a0.w;
    q[j][4] = a1.x; q[j][5] = a1.y; q[j][6] = a1.z; q[j][7] = a1.w;
  }

  const int key0 = c * kAttnChunk + warp * 32;
  uint4 kr[ITER][LOADS];
#pragma unroll
  for (int it = 0; it < ITER; ++it) {
    const int key = key0 + it * 8 + g;
#pragma unroll
    for (int j = 0; j < LOADS; ++j)
      kr[it][j] = (key < n) ? ld_stream(Kh + (size_t)key * DH + (j * 4 + qd) * 8)
                            : make_uint4(0, 0, 0, 0);
  }
  float sc[ITER];
#pragma unroll
  for (int it = 0; it < ITER; ++it) {
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < LOADS; ++j) {
      float kf[8];
      unpack8(kr[it][j], kf);
#pragma unroll
      for (int t = 0; t < 8; ++t) dot = fmaf(q[j][t], kf[t], dot);
    }
    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
    dot += __shfl_xor_sync(0xffffffffu, dot, 2);
    sc[it] = (key0 + it * 8 + g < n) ? dot * a.q_scale : -INFINITY;
  }
  float m = sc[0];
#pragma unroll
  for (int it = 1; it < ITER; ++it) m = fmaxf(m, sc[it]);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

  __shared__ float sm_m[kAttnWarps], sm_l[kAttnWarps];
  __shared__ float sm_o[kAttnWarps][DH];
  __shared__ int sm_last;

  float l = 0.f;
  float acc[LOADS][8];
#pragma unroll
  for (int j = 0; j < LOADS; ++j)
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[j][t] = 0.f;
  if (m != -INFINITY) {   // warp-uniform: this warp has at least one valid key
    float p[ITER];
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
      p[it] = (sc[it] == -INFINITY) ? 0.f : exp2f(sc[it] - m);
      l += p[it];
    }
    uint4 vr[ITER][LOADS];
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
      const int key = key0 + it * 8 + g;
#pragma unroll
      for (int j = 0; j < LOADS; ++j)
        vr[it][j] = (key < n) ? ld_stream(Vh + (size_t)key * DH + (j * 4 + qd) * 8)
                              : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
#pragma unroll
      for (int j = 0; j < LOADS; ++j) {
        float vf[8];
        unpack8(vr[it][j], vf);
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[j][t] = fmaf(p[it], vf[t], acc[j][t]);
      }
    }
  }
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
    for (int j = 0; j < LOADS; ++j)
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[j][t] += __shfl_xor_sync(0xffffffffu, acc[j][t], o);
  }
  if (lane == 0) { sm_m[warp] = m; sm_l[warp] = l; }
  if (g == 0) {
#pragma unroll
    for (int j = 0; j < LOADS; ++j)
#pragma unroll
      for (int t = 0; t < 8; ++t) sm_o[warp][(j * 4 + qd) * 8 + t] = acc[j][t];
  }
  __syncthreads();

  // chunk partial: merge the warps in warp order
  float* part = a.part + (((size_t)s * a.H + h) * a.nc_max) * (DH + 2);
  {
    float M = sm_m[0];
    for (int w = 1; w < kAttnWarps; ++w) M = fmaxf(M, sm_m[w]);
    for (int i = threadIdx.x; i < DH + 1; i += blockDim.x) {
      float v = 0.f;
      for (int w = 0; w < kAttnWarps; ++w) {
        const float f = (sm_m[w] == -INFINITY) ? 0.f : exp2f(sm_m[w] - M);
        v = fmaf(f, (i < DH) ? sm_o[w][i] : sm_l[w], v);
      }
      float* dst = part + (size_t)c * (DH + 2);
      if (i < DH) dst[2 + i] = v; else dst[1] = v;
      if (i == 0) dst[0] = M;
    }
  }
  __threadfence();
  __syncthreads();
  pdl_trigger();   // this chunk is done: the next kernel may start launching
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(a.count + (size_t)s * a.H + h, 1u);
    sm_last = (prev == (unsigned)(nc - 1));
  }
  __syncthreads();
  if (!sm_last) return;
  __threadfence();

  // last CTA: merge the chunks in chunk order
  float M = -INFINITY;
  for (int cc = 0; cc < nc; ++cc) M = fmaxf(M, __ldcg(part + (size_t)cc * (DH + 2)));
  for (int i = threadIdx.x; i < DH; i += blockDim.x) {
    float L = 0.f, O = 0.f;
    for (int cc = 0; cc < nc; ++cc) {
      const float* src = part + (size_t)cc * (DH + 2);
      const float f = exp2f(__ldcg(src) - M);
      L = fmaf(f, __ldcg(src + 1), L);
      O = fmaf(f, __ldcg(src + 2 + i), O);
    }
    o_out[i] = O / L;
    if (a.op) op_store(a.op, HD, a.op_Bp, s, h * DH + i, O / L);
  }
  if (threadIdx.x == 0) a.count[(size_t)s * a.H + h] = 0u;
}

}  // namespace

cudaError_t launch_attn_args(const AttnArgs& a, int B, int Dh, cudaStream_t s) {
  const dim3 grid(a.nc_max, a.H, B);
  switch (Dh) {
    case 32: return launch_k(k_attn<32>, grid, dim3(kAttnWarps * 32), 0, s, 1, a);
    case 64: return launch_k(k_attn<64>, grid, dim3(kAttnWarps * 32), 0, s, 1, a);
    case 128: return launch_k(k_attn<128>, grid, dim3(kAttnWarps * 32), 0, s, 1, a);
    default: return cudaErrorInvalidValue;
  }
}

// The tick's attention for one layer: the slot's rotated, pre-scaled q against its ring.
cudaError_t launch_attn(const Dims& D, const Buffers& b, int layer, bool op, cudaStream_t s) {
  AttnArgs a{};
  a.q = b.q;
  a.q_ld = D.d;
  a.q_scale = 1.0f;   // q already carries log2(e) / sqrt(Dh)
  const size_t blk = (size_t)D.W * D.Dh;
  a.k = b.ring + ((size_t)layer * D.B * 2 + 0) * D.H * blk;
  a.v = a.k + (size_t)D.H * blk;
  a.slot_stride = 2 * (size_t)D.H * blk;
  a.n_valid = b.nvalid;
  a.H = D.H;
  a.W = D.W;
  a.nc_max = D.nc_max;
  a.out = b.o;
  a.out_ld = D.d;
  a.op = op ? b.op_o : nullptr;
  a.op_Bp = D.Bp;
  a.part = b.attn_part;
  a.count = b.attn_count;
  return launch_attn_args(a, D.B, D.Dh, s);
}

}  // namespace pp
