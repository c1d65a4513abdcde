// k_dep_persist.cu - the depformer's 16 codebook steps as one persistent kernel, for
// small batches (PP_FLAG_LOW_LATENCY, up to kPMaxB slots).
//
// The depformer is 16 autoregressive steps of 6 layers each; launched one contraction
// at a time it is ~300 dependent kernels per tick, each paying a launch, its first loads
// and its epilogue.  Here one cooperative launch (one CTA per SM, all co-resident) runs
// every phase of every step and separates phases with a grid barrier:
//   step k:  in-projection  y = P_k z + D_k[tok]                       (z = final-norm x)
//            per layer j:   qkv = W_qkv RMSNorm(y)        | attention over steps 0..k
//                           y += W_o o                    | h = silu(W_g n) * (W_u n)
//                           y += W_down h                 (n = RMSNorm(y))
//            head           logits_k = H_k RMSNorm(y); row k+1 = argmax (agent rows,
//                           unless forced) or the user code (user rows)
// Contractions run on the CUDA cores in fp32: every CTA stages the phase's input vectors
// (normalised where the phase takes a norm, each CTA computing the same sums in the same
// order) in shared memory, and each warp computes whole weight rows, lane-strided 16-byte
// chunks added in chunk order and then over a fixed shuffle tree.  Every result depends
// on the weights, the slot's own inputs and the device's SM count only, never on the
// batch.  After the head every CTA reduces the per-CTA argmax partials itself, so the
// next step starts without another barrier.
// Every barrier wait is bounded: on expiry the kernel raises PP_S_TIMEOUT, marks a
// global abort that the other CTAs see at their next barrier, and every CTA returns.
#include <math.h>

#include "pp_async.cuh"
#include "pp_attn_common.cuh"
#include "pp_internal.cuh"

namespace pp {

namespace {

constexpr int kPThreads = 512;
constexpr int kPWarps = kPThreads / 32;

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// the greedy order: a larger value, or an equal value at a lower index (NaN never wins)
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

struct Shared {
  int tok[kPMaxB];         // token feeding the current step
  int live[kPMaxB];
  float rstd[kPMaxB];
  float red[kPWarps][kPMaxB];
  float amv[kPWarps][kPMaxB];   // per-warp argmax value / index of the head phase
  int ami[kPWarps][kPMaxB];
  int amn[kPWarps];             // a NaN was seen
  int abort;
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void red_add_release(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid barrier on (count, gen): thread 0 of each CTA arrives with a release (after the
// CTA barrier, so it releases every thread's writes); the last to arrive resets the
// count and advances the generation with a release; the others poll the generation
// with acquire loads, spinning first and then sleeping.  Bounded: a CTA that waits
// longer than the budget raises the timeout and the global abort; a CTA that sees the
// abort stops too.  Returns false to stop.
__device__ bool grid_sync(const PersistArgs& p, Shared& sh, uint32_t budget, bool leave = false) {
  __syncthreads();
  if (leave) return false;   // a failure-detection test: this CTA never arrives
  if (threadIdx.x == 0) {
    const unsigned g = ld_acquire(p.bar_gen);
    if (atom_add_acq_rel(p.bar_count, 1u) == gridDim.x - 1) {
      *reinterpret_cast<volatile unsigned*>(p.bar_count) = 0u;
      red_add_release(p.bar_gen, 1u);
    } else {
      uint32_t i = 0;
      while (ld_acquire(p.bar_gen) == g) {
        if (++i < 512) continue;   // spin first: a phase ends within microseconds
        if (*reinterpret_cast<volatile int*>(p.abort)) { sh.abort = 1; break; }
        if (i > budget) {
          sh.abort = 1;
          atomicExch(p.abort, 1);
          atomicOr(p.b.status, PP_S_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
    }
    if (*reinterpret_cast<volatile int*>(p.abort)) sh.abort = 1;
  }
  __syncthreads();
  return !sh.abort;
}

// L2 prefetch of this warp's rows of the next phase's matrix (rows m = gw, gw + GW, ...;
// with `pair`, also row pair + m): issued a phase ahead so that the next phase's row
// loads meet L2 rather than HBM
__device__ __forceinline__ void prefetch_rows(const uint16_t* W, int M, int K, int pair, int gw,
                                              int GW) {
  if ((threadIdx.x & 31) != 0) return;
  const uint32_t bytes = (uint32_t)K * 2;   // a multiple of 16 (K % 8 == 0)
  for (int m = gw; m < M; m += GW) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(W + (size_t)m * K), "r"(bytes)
                 : "memory");
    if (pair)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(W + (size_t)(pair + m) * K),
                   "r"(bytes)
                   : "memory");
  }
}

// dot products of weight row `row` (K bf16, 16-byte aligned) with the B staged vectors
// xs[b][K] (fp32, shared): lane l adds the chunks l, l+32, ... in order (8 chunk loads in
// flight before any is used), then the lanes are added over a fixed shuffle tree; every
// lane returns the B sums
template <int MAXB>
__device__ __forceinline__ void row_dots(const uint16_t* __restrict__ w, int K, const float* xs,
                                         int B, float out[MAXB]) {
  constexpr int kBatch = 8;
  const int lane = threadIdx.x & 31;
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  const int nch = K >> 3;
#pragma unroll
  for (int b = 0; b < MAXB; ++b) out[b] = 0.f;
  for (int c0 = lane; c0 < nch; c0 += 32 * kBatch) {
    uint4 wv[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int c = c0 + 32 * i;
      wv[i] = c < nch ? __ldg(wr + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int c = c0 + 32 * i;
      if (c >= nch) break;
      const float f[8] = {bf16lo(wv[i].x), bf16hi(wv[i].x), bf16lo(wv[i].y), bf16hi(wv[i].y),
                          bf16lo(wv[i].z), bf16hi(wv[i].z), bf16lo(wv[i].w), bf16hi(wv[i].w)};
#pragma unroll
      for (int b = 0; b < MAXB; ++b) {
        if (b < B) {
          const float* x = xs + (size_t)b * K + (c << 3);
          float a = out[b];
#pragma unroll
          for (int e = 0; e < 8; ++e) a = fmaf(f[e], x[e], a);
          out[b] = a;
        }
      }
    }
  }
#pragma unroll
  for (int b = 0; b < MAXB; ++b)
    if (b < B)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) out[b] += __shfl_xor_sync(0xffffffffu, out[b], o);
}

// Stage src[b][0..K) (global, written by other CTAs: read through L2) into xs[b][K],
// optionally as RMSNorm(src[b]) * alpha.  Every CTA computes the same sums in the same
// order: thread t adds elements t, t + kPThreads, ... then the warps' sums are added in
// warp order.
__device__ void stage(const float* src, int ld, int K, int B, const float* alpha, float eps,
                      float* xs, Shared& sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int b = 0; b < B; ++b) {
    float ss = 0.f;
    for (int i = threadIdx.x; i < K; i += kPThreads) {
      const float v = __ldcg(src + (size_t)b * ld + i);
      xs[(size_t)b * K + i] = v;
      ss = fmaf(v, v, ss);
    }
    if (alpha) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) sh.red[warp][b] = ss;
    }
  }
  __syncthreads();
  if (!alpha) return;
  if (threadIdx.x < B) {
    float t = 0.f;
    for (int w = 0; w < kPWarps; ++w) t += sh.red[w][threadIdx.x];
    sh.rstd[threadIdx.x] = 1.0f / sqrtf(t / (float)K + eps);
  }
  __syncthreads();
  for (int b = 0; b < B; ++b) {
    const float r = sh.rstd[b];
    for (int i = threadIdx.x; i < K; i += kPThreads) xs[(size_t)b * K + i] *= r * alpha[i];
  }
  __syncthreads();
}

template <int MAXB>
__global__ void __launch_bounds__(kPThreads, 1) k_dep_persist(const PersistArgs p) {
  extern __shared__ __align__(16) float xs[];   // [B][max(d, Fd)] staged input vectors
  __shared__ Shared sh;
  const Dims& D = p.D;
  const Buffers& b = p.b;
  const int B = D.B, dd = D.dd, Fd = D.Fd, Va = D.Va, nq = D.nq;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kPWarps + warp, GW = gridDim.x * kPWarps;
  const uint32_t budget = wait_budget(b.test_ctl);
  pdl_wait_and_trigger();
  __shared__ int s_leave;
  if (threadIdx.x == 0) {
    sh.abort = 0;
    int32_t armed, kinds;
    read_withhold(b.test_ctl, armed, kinds);
    s_leave = take_withhold(b.test_ctl, armed, kinds, PP_TEST_PERSIST) ? 1 : 0;
  }
  if (threadIdx.x < B) {
    sh.tok[threadIdx.x] = b.tok[threadIdx.x];    // the frame's text token (or forced)
    sh.live[threadIdx.x] = b.live[threadIdx.x];
  }
  __syncthreads();
  float v[MAXB];
  for (int k = 0; k < nq; ++k) {
    // ---- in-projection: y = P_k z + D_k[tok], z = x * rstd_z * out_alpha ------------
    prefetch_rows(b.dep_wqkv, 3 * dd, dd, 0, gw, GW);   // layer 0's qkv
    for (int bb = 0; bb < B; ++bb) {
      const float r = b.rstd_z[bb];
      for (int i = threadIdx.x; i < D.d; i += kPThreads)
        xs[(size_t)bb * D.d + i] = __ldcg(b.x + (size_t)bb * D.d + i) * r * b.out_alpha[i];
    }
    __syncthreads();
    {
      const uint16_t* P = b.dep_inproj + (size_t)k * dd * D.d;
      const uint16_t* E = (k == 0) ? b.dep_emb_text
                                   : b.dep_emb_audio + (size_t)(k - 1) * (Va + 1) * dd;
      for (int m = gw; m < dd; m += GW) {
        row_dots<MAXB>(P + (size_t)m * D.d, D.d, xs, B, v);
        if (lane < B) {
          float val = v[0];
#pragma unroll
          for (int bb = 1; bb < MAXB; ++bb)
            if (bb == lane) val = v[bb];
          const uint16_t e = E[(size_t)sh.tok[lane] * dd + m];
          b.y[(size_t)lane * dd + m] = val + __uint_as_float((uint32_t)e << 16);
        }
      }
    }
    if (!grid_sync(p, sh, budget, k == 0 && s_leave)) return;
    for (int j = 0; j < D.Ld; ++j) {
      // ---- qkv = W_qkv RMSNorm(y) ------------------------------------------------------
      prefetch_rows(b.dep_wo + (size_t)j * dd * dd, dd, dd, 0, gw, GW);   // for the o-proj
      stage(b.y, dd, dd, B, b.dep_attn_alpha + (size_t)j * dd, D.eps, xs, sh);
      {
        const uint16_t* W = b.dep_wqkv + (size_t)j * 3 * dd * dd;
        for (int m = gw; m < 3 * dd; m += GW) {
          row_dots<MAXB>(W + (size_t)m * dd, dd, xs, B, v);
#pragma unroll
          for (int bb = 0; bb < MAXB; ++bb)
            if (bb < B && lane == bb) b.dqkv[(size_t)bb * 3 * dd + m] = v[bb];
        }
      }
      if (!grid_sync(p, sh, budget)) return;
      // ---- attention of step k over the frame's steps 0..k (one warp per slot, head) ----
      // lane t scores key t (a sequential dot over the head's dims), the lanes take the
      // softmax over a fixed shuffle tree, then each lane adds p_t v_t over t in order
      // for its own dims; every load of a step is issued before its first use
      for (int task = gw; task < B * D.Hd; task += GW) {
        const int s = task / D.Hd, h = task - s * D.Hd;
        const float* row = b.dqkv + (size_t)s * 3 * dd + h * D.Dhd;
        float* cache = b.dkv + ((size_t)s * D.Ld + j) * nq * 2 * dd;
        for (int i = lane; i < D.Dhd; i += 32) {
          cache[(size_t)k * 2 * dd + h * D.Dhd + i] = __ldcg(row + dd + i);
          cache[(size_t)k * 2 * dd + dd + h * D.Dhd + i] = __ldcg(row + 2 * dd + i);
        }
        __syncwarp();
        float sc = -INFINITY;
        if (lane <= k) {
          const float4* q4 = reinterpret_cast<const float4*>(row);
          const float4* k4 = reinterpret_cast<const float4*>(cache + (size_t)lane * 2 * dd + h * D.Dhd);
          float dot = 0.f;
          for (int i = 0; i < (D.Dhd >> 2); ++i) {
            const float4 a = __ldcg(q4 + i), c = __ldcg(k4 + i);
            dot = fmaf(a.x, c.x, dot);
            dot = fmaf(a.y, c.y, dot);
            dot = fmaf(a.z, c.z, dot);
            dot = fmaf(a.w, c.w, dot);
          }
          sc = dot * (1.0f / sqrtf((float)D.Dhd));
        }
        float mx = sc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float pw = lane <= k ? expf(sc - mx) : 0.f;
        float l = pw;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        for (int i = lane; i < D.Dhd; i += 32) {
          float vt[16];
#pragma unroll
          for (int t = 0; t < 16; ++t)
            vt[t] = t <= k ? __ldcg(cache + (size_t)t * 2 * dd + dd + h * D.Dhd + i) : 0.f;
          float acc = 0.f;
#pragma unroll
          for (int t = 0; t < 16; ++t) acc = fmaf(__shfl_sync(0xffffffffu, pw, t), vt[t], acc);
          b.dout[(size_t)s * dd + h * D.Dhd + i] = acc / l;
        }
      }
      if (!grid_sync(p, sh, budget)) return;
      // ---- y += W_o o ----------------------------------------------------------------------
      prefetch_rows(b.dep_wgu + (size_t)j * 2 * Fd * dd, Fd, dd, Fd, gw, GW);   // gate/up
      stage(b.dout, dd, dd, B, nullptr, 0.f, xs, sh);
      {
        const uint16_t* W = b.dep_wo + (size_t)j * dd * dd;
        for (int m = gw; m < dd; m += GW) {
          row_dots<MAXB>(W + (size_t)m * dd, dd, xs, B, v);
#pragma unroll
          for (int bb = 0; bb < MAXB; ++bb)
            if (bb < B && lane == bb) b.y[(size_t)bb * dd + m] = __ldcg(b.y + (size_t)bb * dd + m) + v[bb];
        }
      }
      if (!grid_sync(p, sh, budget)) return;
      // ---- h = silu(W_g n) * (W_u n), n = RMSNorm(y) ---------------------------------------
      prefetch_rows(b.dep_wdown + (size_t)j * dd * Fd, dd, Fd, 0, gw, GW);   // for the down
      stage(b.y, dd, dd, B, b.dep_mlp_alpha + (size_t)j * dd, D.eps, xs, sh);
      {
        const uint16_t* W = b.dep_wgu + (size_t)j * 2 * Fd * dd;
        float u[MAXB];
        for (int m = gw; m < Fd; m += GW) {
          row_dots<MAXB>(W + (size_t)m * dd, dd, xs, B, v);
          row_dots<MAXB>(W + (size_t)(Fd + m) * dd, dd, xs, B, u);
#pragma unroll
          for (int bb = 0; bb < MAXB; ++bb)
            if (bb < B && lane == bb)
              b.dh[(size_t)bb * Fd + m] = v[bb] / (1.0f + expf(-v[bb])) * u[bb];
        }
      }
      if (!grid_sync(p, sh, budget)) return;
      // ---- y += W_down h ---------------------------------------------------------------------
      if (j + 1 < D.Ld)   // the next layer's qkv, or this step's head
        prefetch_rows(b.dep_wqkv + (size_t)(j + 1) * 3 * dd * dd, 3 * dd, dd, 0, gw, GW);
      else
        prefetch_rows(b.dep_heads + (size_t)k * Va * dd, Va, dd, 0, gw, GW);
      stage(b.dh, Fd, Fd, B, nullptr, 0.f, xs, sh);
      {
        const uint16_t* W = b.dep_wdown + (size_t)j * dd * Fd;
        for (int m = gw; m < dd; m += GW) {
          row_dots<MAXB>(W + (size_t)m * Fd, Fd, xs, B, v);
#pragma unroll
          for (int bb = 0; bb < MAXB; ++bb)
            if (bb < B && lane == bb) b.y[(size_t)bb * dd + m] = __ldcg(b.y + (size_t)bb * dd + m) + v[bb];
        }
      }
      if (!grid_sync(p, sh, budget)) return;
    }
    // ---- head k: logits and this CTA's argmax partial per slot --------------------------
    if (k + 1 < nq)   // the next step's in-projection
      prefetch_rows(b.dep_inproj + (size_t)(k + 1) * dd * D.d, dd, D.d, 0, gw, GW);
    stage(b.y, dd, dd, B, b.dep_out_alpha, D.eps, xs, sh);
    {
      const uint16_t* Hk = b.dep_heads + (size_t)k * Va * dd;
      float bv[MAXB];
      int bi[MAXB];
      int nan = 0;
#pragma unroll
      for (int bb = 0; bb < MAXB; ++bb) { bv[bb] = -INFINITY; bi[bb] = 0x7FFFFFFF; }
      for (int m = gw; m < Va; m += GW) {
        row_dots<MAXB>(Hk + (size_t)m * dd, dd, xs, B, v);
#pragma unroll
        for (int bb = 0; bb < MAXB; ++bb) {
          if (bb < B) {
            if (lane == bb) b.logits[(size_t)bb * D.logits_ld + D.Vt + (size_t)k * Va + m] = v[bb];
            if (isnan(v[bb])) nan = 1;
            else if (better(v[bb], m, bv[bb], bi[bb])) { bv[bb] = v[bb]; bi[bb] = m; }
          }
        }
      }
      if (lane == 0) {
#pragma unroll
        for (int bb = 0; bb < MAXB; ++bb) { sh.amv[warp][bb] = bv[bb]; sh.ami[warp][bb] = bi[bb]; }
        sh.amn[warp] = nan;
      }
      __syncthreads();
      if (threadIdx.x < B) {
        const int bb = threadIdx.x;
        float cv = -INFINITY;
        int ci = 0x7FFFFFFF, cn = 0;
        for (int w = 0; w < kPWarps; ++w) {
          if (better(sh.amv[w][bb], sh.ami[w][bb], cv, ci)) { cv = sh.amv[w][bb]; ci = sh.ami[w][bb]; }
          cn |= sh.amn[w];
        }
        p.part_val[(size_t)blockIdx.x * kPMaxB + bb] = cv;
        p.part_idx[(size_t)blockIdx.x * kPMaxB + bb] = ci | (cn ? (int)0x80000000 : 0);
      }
    }
    if (!grid_sync(p, sh, budget)) return;
    // ---- every CTA: the decision of row k+1 from all partials (the same in every CTA) ----
    // warp bb reduces slot bb's partials (lane l takes CTAs l, l+32, ...; the greedy
    // order is a total order, so any reduction tree gives the same token)
    if (warp < B) {
      const int bb = warp, row = k + 1;
      float cv = -INFINITY;
      int ci = 0x7FFFFFFF, cn = 0;
      for (int c = lane; c < (int)gridDim.x; c += 32) {
        const float pv = __ldcg(p.part_val + (size_t)c * kPMaxB + bb);
        const int pi = __ldcg(p.part_idx + (size_t)c * kPMaxB + bb);
        cn |= (pi < 0);
        const int idx = pi & 0x7FFFFFFF;
        if (better(pv, idx, cv, ci)) { cv = pv; ci = idx; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, cv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, ci, o);
        cn |= __shfl_xor_sync(0xffffffffu, cn, o);
        if (better(ov, oi, cv, ci)) { cv = ov; ci = oi; }
      }
      if (lane == 0) {
        if (ci == 0x7FFFFFFF) ci = 0;   // every logit NaN
        int t;
        if (row <= PP_AGENT_ROWS)
          t = b.in_fmask[bb * kRows + row] ? b.in_forced[bb * kRows + row] : ci;
        else
          t = b.in_user[bb * PP_USER_ROWS + row - 1 - PP_AGENT_ROWS];
        const bool bad = t < 0 || t > Va;
        if (bad) t = Va;
        if (!sh.live[bb]) t = 0;
        sh.tok[bb] = t;
        if (blockIdx.x == 0) {
          b.out_col[bb * kRows + row] = sh.live[bb] ? t : -1;
          if (sh.live[bb]) {
            if (bad) atomicOr(b.status, PP_S_INDEX);
            if (cn && row <= PP_AGENT_ROWS && !b.in_fmask[bb * kRows + row])
              atomicOr(b.status, PP_S_NAN);
          }
        }
      }
    }
    __syncthreads();
  }
}

}  // namespace

int persist_grid() { return attn::sm_count(); }

size_t persist_smem(const Dims& D) {
  const int wide = D.d > D.Fd ? D.d : D.Fd;
  return (size_t)D.B * wide * sizeof(float);
}

cudaError_t persist_setup(const Dims& D) {
  const size_t smem = persist_smem(D);
  if (D.B > kPMaxB || smem > 200 * 1024) return cudaErrorInvalidValue;
  return cudaFuncSetAttribute(k_dep_persist<kPMaxB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem);
}

cudaError_t launch_dep_persist(const PersistArgs& p, cudaStream_t s) {
  const int grid = persist_grid();
  if (grid > kPMaxGrid) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = persist_smem(p.D);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: the grid barrier is safe
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_dep_persist<kPMaxB>, p);
}

}  // namespace pp
