// k_attn.cu - split-K sliding-window decode attention over each slot's ring KV.
//
// For slot s at position p the valid ring indices are 0 .. n-1 with n = min(p+1, W):
// before the ring wraps they hold positions 0..p in place, after it every index holds
// one of the last W positions.  Softmax is invariant to the order of its keys, so the
// kernel attends over ring indices directly.
//
// Work unit = (slot, head, chunk of kAttnChunk consecutive ring indices).  The kernel is
// persistent: one CTA per SM walks the units u = blockIdx.x, + gridDim.x, ... and skips
// chunks past a slot's n.  Per CTA:
//   warp 8 lane 0   producer: bulk-copies each unit's K rows, V rows and the head's
//                   query into a ring of shared-memory stages (mbarrier transaction
//                   counts), so the HBM stream never waits on arithmetic;
//   warps 0-3, 4-7  two consumer warpgroups taking alternate units.  Each warp scores
//                   32 keys (4 lanes per key, 16-byte pieces XOR-swizzled by key parity
//                   so that a quarter-warp's shared loads hit distinct banks), then
//                   accumulates p.V with each lane owning Dh/32 output dims.  The four
//                   warp partials are merged in warp order into the chunk partial
//                   (max, sum, unnormalised output), written to global scratch; the
//                   last unit of a (slot, head) to finish merges the chunks in chunk
//                   order.
// Every reduction order is fixed by ring index alone, so a slot's result does not depend
// on the other slots, on the grid or on timing.
#include <math.h>

#include "pp_async.cuh"
#include "pp_attn_common.cuh"
#include "pp_internal.cuh"

namespace pp {

namespace {

using namespace attn;

constexpr int kConsumerWarps = 8;                      // each takes 16 keys of a unit
constexpr int kKeysPerWarp = kAttnChunk / kConsumerWarps;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kEpilogueWarp = kConsumerWarps + 1;
constexpr int kAttnThreads = (kConsumerWarps + 2) * 32;
constexpr int kPartSlots = 4;                          // warp-partial slots in flight
static_assert(kKeysPerWarp % 8 == 0, "8 keys per score iteration");

template <int DH>
struct AttnCfg {
  static constexpr int kKVBytes = kAttnChunk * DH * 2;          // K (or V) rows of one unit
  static constexpr int kStageBytes = 2 * kKVBytes + DH * 4;     // K, V, fp32 query
  static constexpr int kWarpPart = DH + 4;                      // m, l, -, -, o[DH] (floats)
  static constexpr int kSlotBytes = kConsumerWarps * kWarpPart * 4;
  static constexpr int kStagesRaw = (196 * 1024) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
  // stages | warp-partial slots | p [8][16] | barriers | flags
  static constexpr int kSlotOff = kStages * kStageBytes;
  static constexpr int kPOff = kSlotOff + kPartSlots * kSlotBytes;
  static constexpr int kBarOff = kPOff + kConsumerWarps * kKeysPerWarp * 4;
  static constexpr int kNumBars = 3 * kStages + 2 * kPartSlots;
  static constexpr int kFlagOff = kBarOff + kNumBars * 8;
  static constexpr int kSmem = kFlagOff + 16;
  static_assert(kStages >= 2, "attention stage does not fit shared memory");
  static_assert(kSmem <= 227 * 1024, "attention shared memory");
  static_assert(kStageBytes % 16 == 0 && kSlotBytes % 16 == 0, "16-byte alignment");
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
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

// DPL consecutive bf16 values at a 2*DPL-byte aligned shared address, as fp32.
template <int DPL>
__device__ __forceinline__ void lds_dims(const uint16_t* p, float f[DPL]) {
  if constexpr (DPL == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  } else if constexpr (DPL == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    f[0] = __uint_as_float(w << 16);
    f[1] = __uint_as_float(w & 0xFFFF0000u);
  } else {
    f[0] = __uint_as_float((uint32_t)*p << 16);
  }
}

// DPL floats at a 4*DPL-byte aligned address (shared or global)
template <int DPL>
__device__ __forceinline__ void ld_f(const float* p, float f[DPL]) {
  if constexpr (DPL == 4) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
  } else if constexpr (DPL == 2) {
    const float2 x = *reinterpret_cast<const float2*>(p);
    f[0] = x.x; f[1] = x.y;
  } else {
    f[0] = *p;
  }
}
template <int DPL>
__device__ __forceinline__ void st_f(float* p, const float f[DPL]) {
  if constexpr (DPL == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  } else if constexpr (DPL == 2) {
    *reinterpret_cast<float2*>(p) = make_float2(f[0], f[1]);
  } else {
    *p = f[0];
  }
}

template <int DH>
__global__ void __launch_bounds__(kAttnThreads, 1) k_attn(AttnArgs a, int units) {
  using C = AttnCfg<DH>;
  constexpr int S = C::kStages;
  constexpr int PIECES = DH / 8;        // 16-byte pieces per K row
  constexpr int LOADS = PIECES / 4;     // pieces per lane (4 lanes per key)
  constexpr int DPL = DH / 32;          // output dims per lane in p.V and in the merges
  constexpr int ITER = kKeysPerWarp / 8;
  static_assert(PIECES % 4 == 0, "head dim must be a multiple of 32");
  extern __shared__ __align__(128) uint8_t smem[];
  float* s_slot = reinterpret_cast<float*>(smem + C::kSlotOff);
  float* s_p = reinterpret_cast<float*>(smem + C::kPOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  // bars: [0,S) K+q full | [S,2S) V full | [2S,3S) stage empty | [3S,3S+P) slot full |
  //       [3S+P,3S+2P) slot empty
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kFlagOff);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t blk = (size_t)a.W * DH;
  // this CTA's contiguous range of units
  const int u0 = (int)(((long long)blockIdx.x * units) / gridDim.x);
  const int u1 = (int)(((long long)(blockIdx.x + 1) * units) / gridDim.x);

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(bar(i), 1);
      mbar_init(bar(S + i), 1);
      mbar_init(bar(2 * S + i), kConsumerWarps);
    }
    for (int i = 0; i < kPartSlots; ++i) {
      mbar_init(bar(3 * S + i), kConsumerWarps);
      mbar_init(bar(3 * S + kPartSlots + i), 1);
    }
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait_and_trigger();

  if (warp == kProducerWarp) {
    // ---- producer -----------------------------------------------------------------
    if (lane == 0) {
      int32_t armed, kinds;
      read_withhold(a.test_ctl, armed, kinds);
      int v = 0;
      for (int u = u0; u < u1; ++u) {
        const Unit t = decode_unit(a, u);
        if (t.nk == 0) continue;
        const int st = v % S;
        if (v >= S && !mbar_wait(bar(2 * S + st), ((v / S) - 1) & 1, a.test_ctl))
          raise_timeout(a, s_abort);
        if (*s_abort) break;
        uint8_t* sk = smem + st * C::kStageBytes;
        const size_t off = (size_t)t.s * a.slot_stride + t.h * blk + (size_t)t.c * kAttnChunk * DH;
        const uint32_t bytes = (uint32_t)t.nk * DH * 2;
        mbar_expect_tx(bar(st), bytes + DH * 4);
        bulk_load(smem_u32(sk), a.k + off, bytes, bar(st));
        bulk_load(smem_u32(sk + 2 * C::kKVBytes), a.q + (size_t)t.s * a.q_ld + t.h * DH, DH * 4,
                  bar(st));
        // a failure-detection test may have this producer withhold its first V tile:
        // that stage never completes and the consumers' bounded waits run out
        if (!(v == 0 && take_withhold(a.test_ctl, armed, kinds, PP_TEST_ATTN))) {
          mbar_expect_tx(bar(S + st), bytes);
          bulk_load(smem_u32(sk + C::kKVBytes), a.v + off, bytes, bar(S + st));
        }
        ++v;
      }
      // every copy this CTA issued lands before the CTA may exit (bounded waits)
      for (int i = v > S ? v - S : 0; i < v; ++i) {
        mbar_wait(bar(i % S), (i / S) & 1, a.test_ctl);
        mbar_wait(bar(S + i % S), (i / S) & 1, a.test_ctl);
      }
    }
    return;
  }

  if (warp == kEpilogueWarp) {
    // ---- epilogue: warp partials -> chunk partial; tickets; final merges -----------
    const int HD = a.H * DH;
    int v = 0, run_pair = -1, run_len = 0, run_nc = 0;
    auto flush = [&]() {   // this CTA's chunks of run_pair are all written
      if (run_len == 0) return;
      __syncwarp();
      unsigned last = 0;
      if (lane == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(a.count + run_pair, (unsigned)run_len);
        last = (prev + (unsigned)run_len == (unsigned)run_nc);
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence();
        const int s = run_pair / a.H, h = run_pair - s * a.H;
        merge_pair<DH>(a, a.part + (size_t)run_pair * attn_pair_floats(a.nc_max, DH), run_nc, s,
                       h, lane);
        if (lane == 0) a.count[run_pair] = 0u;
      }
      run_len = 0;
    };
    for (int u = u0; u < u1; ++u) {
      const Unit t = decode_unit(a, u);
      const int pair = t.s * a.H + t.h;
      if (t.nk == 0) {
        if (t.c == 0) {   // closed slot: zero output
          for (int i = lane; i < DH; i += 32) {
            a.out[(size_t)t.s * a.out_ld + t.h * DH + i] = 0.f;
            if (a.op) op_store(a.op, HD, a.op_Bp, t.s, t.h * DH + i, 0.f);
          }
        }
        continue;
      }
      if (pair != run_pair) {
        flush();
        run_pair = pair;
        run_nc = (min(__ldg(a.n_valid + t.s), a.W) + kAttnChunk - 1) / kAttnChunk;
      }
      const int ps = v % kPartSlots;
      const uint32_t ph = (v / kPartSlots) & 1;
      ++v;
      if (!*s_abort && !mbar_wait(bar(3 * S + ps), ph, a.test_ctl)) raise_timeout(a, s_abort);
      const float* slot = s_slot + ps * (kConsumerWarps * C::kWarpPart);
      float mw[kConsumerWarps];
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        mw[w] = slot[w * C::kWarpPart];
        M = fmaxf(M, mw[w]);
      }
      float L = 0.f, O[DPL];
#pragma unroll
      for (int i = 0; i < DPL; ++i) O[i] = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {   // warp order
        const float f = (mw[w] == -INFINITY) ? 0.f : exp2f(mw[w] - M);
        float ow[DPL];
        ld_f<DPL>(slot + w * C::kWarpPart + 4 + lane * DPL, ow);
        L = fmaf(f, slot[w * C::kWarpPart + 1], L);
#pragma unroll
        for (int i = 0; i < DPL; ++i) O[i] = fmaf(f, ow[i], O[i]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(3 * S + kPartSlots + ps));   // slot free
      float* dst = a.part + (size_t)pair * attn_pair_floats(a.nc_max, DH) +
                   (size_t)t.c * attn_rec_floats(DH);
      if (lane < 8) dst[lane] = lane == 0 ? M : (lane == 1 ? L : 0.f);   // whole sector
      st_f<DPL>(dst + 8 + lane * DPL, O);
      ++run_len;
    }
    flush();
    pdl_trigger();
    return;
  }

  // ---- consumers: warp w scores keys w*16 .. w*16+15 of each unit, then p.V --------
  const int g = lane >> 2, qd = lane & 3;
  const int par = (LOADS >= 2) ? (g & 1) : 0;   // piece swizzle of this lane's key
  float* pw = s_p + warp * kKeysPerWarp;
  const int key0 = warp * kKeysPerWarp;
  int v = 0;
  for (int u = u0; u < u1; ++u) {
    const Unit t = decode_unit(a, u);
    if (t.nk == 0) continue;
    const int st = v % S, ps = v % kPartSlots;
    const uint32_t ph = (v / S) & 1;
    const bool reuse_slot = v >= kPartSlots;
    const uint32_t pph = ((v / kPartSlots) - 1) & 1;
    ++v;
    const uint8_t* sk = smem + st * C::kStageBytes;
    const uint32_t k_base = smem_u32(sk);
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(sk + C::kKVBytes);
    const float* qs = reinterpret_cast<const float*>(sk + 2 * C::kKVBytes);
    const int kcount = max(0, min(kKeysPerWarp, t.nk - key0));

    if (!*s_abort && !mbar_wait(bar(st), ph, a.test_ctl)) raise_timeout(a, s_abort);
    // scores: lane (g, qd) holds pieces (j ^ par) * 4 + qd of the query and of its key
    float q[LOADS][8];
#pragma unroll
    for (int j = 0; j < LOADS; ++j) {
      const float4* p4 = reinterpret_cast<const float4*>(qs + (((j ^ par) * 4 + qd) * 8));
      const float4 a0 = p4[0], a1 = p4[1];
      q[j][0] = a0.x; q[j][1] = a0.y; q[j][2] = a0.z; q[j][3] = a0.w;
      q[j][4] = a1.x; q[j][5] = a1.y; q[j][6] = a1.z; q[j][7] = a1.w;
    }
    float sc[ITER];
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
      const int key = key0 + it * 8 + g;
      uint4 kr[LOADS];
#pragma unroll
      for (int j = 0; j < LOADS; ++j)
        kr[j] = lds128(k_base + (uint32_t)(key * DH + ((j ^ par) * 4 + qd) * 8) * 2);
      float dot = 0.f;
#pragma unroll
      for (int j = 0; j < LOADS; ++j) {
        float kf[8];
        unpack8(kr[j], kf);
#pragma unroll
        for (int e = 0; e < 8; ++e) dot = fmaf(q[j][e], kf[e], dot);
      }
      dot += __shfl_xor_sync(0xffffffffu, dot, 1);
      dot += __shfl_xor_sync(0xffffffffu, dot, 2);
      sc[it] = (key < t.nk) ? dot * a.q_scale : -INFINITY;
    }
    float m = sc[0];
#pragma unroll
    for (int it = 1; it < ITER; ++it) m = fmaxf(m, sc[it]);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

    float l = 0.f;
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    if (!*s_abort && !mbar_wait(bar(S + st), ph, a.test_ctl)) raise_timeout(a, s_abort);
    if (kcount > 0) {   // warp-uniform
#pragma unroll
      for (int it = 0; it < ITER; ++it) {
        const float p = (sc[it] == -INFINITY) ? 0.f : exp2f(sc[it] - m);
        l += p;
        if (qd == 0) pw[it * 8 + g] = p;
      }
      __syncwarp();
      // p.V in key order; lane owns dims lane*DPL .. +DPL
      const uint16_t* vrow = vs + key0 * DH + lane * DPL;
      int k = 0;
      for (; k + 8 <= kcount; k += 8) {
        float vf[8][DPL];
#pragma unroll
        for (int e = 0; e < 8; ++e) lds_dims<DPL>(vrow + (k + e) * DH, vf[e]);
        const float4 p0 = *reinterpret_cast<const float4*>(pw + k);
        const float4 p1 = *reinterpret_cast<const float4*>(pw + k + 4);
        const float pk[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
          for (int i = 0; i < DPL; ++i) acc[i] = fmaf(pk[e], vf[e][i], acc[i]);
      }
      for (; k < kcount; ++k) {
        float vf[DPL];
        lds_dims<DPL>(vrow + k * DH, vf);
        const float pk = pw[k];
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] = fmaf(pk, vf[i], acc[i]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(2 * S + st));   // stage free
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    // warp partial into the unit's slot
    if (reuse_slot && !*s_abort && !mbar_wait(bar(3 * S + kPartSlots + ps), pph, a.test_ctl))
      raise_timeout(a, s_abort);
    float* wp = s_slot + ps * (kConsumerWarps * C::kWarpPart) + warp * C::kWarpPart;
    if (lane == 0) { wp[0] = m; wp[1] = l; }
    st_f<DPL>(wp + 4 + lane * DPL, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(3 * S + ps));
  }
}

template <int DH>
cudaError_t launch_dh(const AttnArgs& a, int B, cudaStream_t s) {
  using C = AttnCfg<DH>;
  cudaError_t err =
      cudaFuncSetAttribute(k_attn<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (err != cudaSuccess) return err;
  const int units = B * a.H * a.nc_max;
  const int nsm = attn::sm_count();
  const int grid = units < nsm ? units : nsm;
  return launch_k(k_attn<DH>, dim3(grid), dim3(kAttnThreads), (size_t)C::kSmem, s, 1, a, units);
}

}  // namespace

cudaError_t launch_attn_cc(const AttnArgs& a, int B, int Dh, cudaStream_t s) {
  if (B < 1 || a.H < 1 || a.nc_max < 1) return cudaErrorInvalidValue;
  switch (Dh) {
    case 32: return launch_dh<32>(a, B, s);
    case 64: return launch_dh<64>(a, B, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn_args(const AttnArgs& a, int B, int Dh, const AttnMaps* maps,
                             int slot_base, cudaStream_t s) {
  if (Dh == 128) {
    if (!maps || !a.q_op) return cudaErrorInvalidValue;
    return launch_attn_tc(a, B, *maps, slot_base, s);
  }
  return launch_attn_cc(a, B, Dh, s);
}

// The tick's attention for one layer: the slot's rotated, pre-scaled q against its ring.
cudaError_t launch_attn(const Dims& D, const Buffers& b, int layer, bool op, const AttnMaps* maps,
                        cudaStream_t s) {
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
  a.status = b.status;
  a.test_ctl = b.test_ctl;
  a.q_op = b.q_op;
  a.early_trigger = D.B <= kEarlyTriggerMaxB;
  // the K/V maps span every layer's ring: slot coordinate = layer * B + slot
  return launch_attn_args(a, D.B, D.Dh, maps, layer * D.B, s);
}

}  // namespace pp
