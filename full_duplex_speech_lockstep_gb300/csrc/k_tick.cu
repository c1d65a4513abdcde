// k_tick.cu - the light kernels of one lockstep tick: control + 17-table embedding
// sum + RoPE angle table, RMSNorm, RoPE + ring-KV write, the token decisions (greedy,
// forced, or sampled per session), the depformer step attention and the end-of-tick
// bookkeeping.
#include <math.h>

#include "pp_internal.cuh"
#include "pp_sample.cuh"

namespace pp {

namespace {

__device__ __forceinline__ void unpack8(const uint4 v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}


// Fixed-order block sum: per-warp butterfly, then warp 0 adds the warp totals in order.
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x == 0) {
    for (int w = 0; w < NT / 32; ++w) t += sh[w];
    sh[NT / 32] = t;
  }
  __syncthreads();
  float r = sh[NT / 32];
  __syncthreads();
  return r;
}

}  // namespace

// ---- control, embedding, RoPE table --------------------------------------------------
// One CTA per slot.  Applies the host's control word (open/close/reset position),
// validates the previous column, sums its 17 embedding rows in fp32 in row order
// (text row first), and tabulates cos/sin of this frame's RoPE angles from fp64.
__global__ void __launch_bounds__(256) k_begin(Dims D, Buffers b, const float* alpha,
                                              uint16_t* op, float* ssq) {
  pdl_wait_and_trigger();
  const int s = blockIdx.x;
  __shared__ int col[kRows];
  __shared__ int live_s, pos_s;
  if (threadIdx.x == 0) {
    const int c = b.ctl[s];
    if (c & 2) {             // (re)open: set the position once, then clear the request
      b.pos[s] = b.ctl_pos[s];
      b.ctl[s] = c & 1;
      b.hist_len[s] = 0;     // a new session starts without text history
    }
    b.live[s] = c & 1;
    live_s = c & 1;
    pos_s = b.pos[s];
    b.nvalid[s] = live_s ? min(pos_s + 1, D.W) : 0;
  }
  // this slot's attention tickets, and the fused decisions' tickets, start the tick at
  // zero (the kernels leave them zero; a tick whose bounded wait gave up may not have)
  for (int h = threadIdx.x; h < D.H; h += blockDim.x) b.attn_count[(size_t)s * D.H + h] = 0u;
  if (s == 0 && threadIdx.x < 4) b.dticket[threadIdx.x] = 0u;
  if (s == 0 && threadIdx.x < 2) b.dnan[threadIdx.x] = 0u;
  if (threadIdx.x < 2) b.dkey[(size_t)threadIdx.x * D.B + s] = 0ull;
  __syncthreads();
  if (threadIdx.x < kRows) {
    const int r = threadIdx.x;
    const int lim = (r == 0) ? D.Vt : D.Va;   // the initial token is the last table row
    int v = b.in_col[s * kRows + r];
    if (v < 0 || v > lim) {
      if (live_s) atomicOr(b.status, PP_S_INDEX);
      v = lim;
    }
    col[r] = v;
  }
  __syncthreads();
  float* x = b.x + (size_t)s * D.d;
  for (int i = threadIdx.x * 8; i < D.d; i += blockDim.x * 8) {
    float acc[8];
    if (!live_s) {
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[t] = 0.f;
    } else {
      float e[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(b.emb_text + (size_t)col[0] * D.d + i)), acc);
      for (int r = 1; r < kRows; ++r) {
        const uint16_t* row = b.emb_audio + ((size_t)(r - 1) * (D.Va + 1) + col[r]) * D.d + i;
        unpack8(__ldg(reinterpret_cast<const uint4*>(row)), e);
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[t] += e[t];
      }
    }
    reinterpret_cast<float4*>(x + i)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    reinterpret_cast<float4*>(x + i)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    if (op) {   // the first layer's fused RMSNorm: operand hi/lo(alpha * x)
#pragma unroll
      for (int t = 0; t < 8; ++t) op_store(op, D.d, D.Bp, s, i + t, alpha[i + t] * acc[t]);
    }
  }
  if (op) {   // and the sum of x^2 (fixed order: per thread, then per warp, then warps)
    __shared__ float sh[9];
    __syncthreads();
    float ss = 0.f;
    for (int i = threadIdx.x; i < D.d; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
    ss = block_sum<256>(ss, sh);
    if (threadIdx.x == 0) ssq[s] = ss;
  }
  // RoPE angles pos * base^(-2i/Dh), evaluated in fp64 and rounded once to fp32
  for (int i = threadIdx.x; i < D.Dh / 2; i += blockDim.x) {
    const double theta =
        (double)pos_s * pow((double)D.rope_base, -2.0 * (double)i / (double)D.Dh);
    double sn, cs;
    sincos(theta, &sn, &cs);
    b.rope_cs[((size_t)s * (D.Dh / 2) + i) * 2] = (float)cs;
    b.rope_cs[((size_t)s * (D.Dh / 2) + i) * 2 + 1] = (float)sn;
  }
}

cudaError_t launch_begin(const Dims& D, const Buffers& b, const float* alpha, uint16_t* op,
                         float* ssq, cudaStream_t s) {
  { cudaError_t e_ = launch_k(k_begin, dim3(D.B), dim3(256), 0, s, 1, D, b, alpha, op, ssq); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// ---- RMSNorm ---------------------------------------------------------------------------
// out[b, i] = x[b, i] / sqrt(mean_j x[b, j]^2 + eps) * alpha[i], one CTA per slot; the
// sum of squares is taken in a fixed order that does not depend on the batch size.
__global__ void __launch_bounds__(512) k_rmsnorm(const float* __restrict__ x, int ldx,
                                                 const float* __restrict__ alpha, int K,
                                                 float eps, float* __restrict__ out, int ldo,
                                                 uint16_t* __restrict__ op, int Bp) {
  pdl_wait_and_trigger();
  __shared__ float sh[17];
  const int b = blockIdx.x;
  const float* xr = x + (size_t)b * ldx;
  float ss = 0.f;
  for (int i = threadIdx.x; i < K; i += 512) ss = fmaf(xr[i], xr[i], ss);
  ss = block_sum<512>(ss, sh);
  const float r = 1.0f / sqrtf(ss / (float)K + eps);
  for (int i = threadIdx.x; i < K; i += 512) {
    const float v = xr[i] * r * alpha[i];
    if (out) out[(size_t)b * ldo + i] = v;
    if (op) op_store(op, K, Bp, b, i, v);
  }
}

cudaError_t launch_rmsnorm(const Dims& D, const float* x, int ldx, const float* alpha, int K,
                           float* out, int ldo, uint16_t* op, cudaStream_t s) {
  { cudaError_t e_ = launch_k(k_rmsnorm, dim3(D.B), dim3(512), 0, s, 1, x, ldx, alpha, K, D.eps, out, ldo, op, D.Bp); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// ---- RoPE + ring write -----------------------------------------------------------------
// One CTA per (slot, head), one thread per rotation pair.  q is rotated and pre-scaled
// by log2(e)/sqrt(Dh) (the attention kernel works in base 2); k is rotated; k and v are
// rounded to bf16 into ring index pos mod W of this layer's ring.
__global__ void k_rope_ring(Dims D, Buffers b, int layer) {
  pdl_wait_and_trigger();
  const int s = blockIdx.x, h = blockIdx.y, i = threadIdx.x;
  if (!b.live[s] || i >= D.Dh / 2) return;
  const int p = b.pos[s];
  const int widx = p % D.W;
  const float c = b.rope_cs[((size_t)s * (D.Dh / 2) + i) * 2];
  const float sn = b.rope_cs[((size_t)s * (D.Dh / 2) + i) * 2 + 1];
  const float* row = b.qkv + (size_t)s * 3 * D.d + h * D.Dh + 2 * i;
  const float q0 = row[0], q1 = row[1];
  const float k0 = row[D.d], k1 = row[D.d + 1];
  const float v0 = row[2 * D.d], v1 = row[2 * D.d + 1];
  const float qs = 1.4426950408889634f / sqrtf((float)D.Dh);
  float* q = b.q + (size_t)s * D.d + h * D.Dh + 2 * i;
  const float qr0 = (q0 * c - q1 * sn) * qs, qr1 = (q0 * sn + q1 * c) * qs;
  q[0] = qr0;
  q[1] = qr1;
  // the same query as the bf16 hi/lo operand rows of the tensor-core attention
  uint16_t* qo = b.q_op + ((size_t)(s * D.H + h) * 2) * D.Dh + 2 * i;
  bf16_split(qr0, qo[0], qo[D.Dh]);
  bf16_split(qr1, qo[1], qo[D.Dh + 1]);
  const float kr0 = k0 * c - k1 * sn, kr1 = k0 * sn + k1 * c;
  const size_t blk = (size_t)D.W * D.Dh;
  const size_t kbase = ((((size_t)layer * D.B + s) * 2 + 0) * D.H + h) * blk;
  const size_t vbase = ((((size_t)layer * D.B + s) * 2 + 1) * D.H + h) * blk;
  const size_t off = (size_t)widx * D.Dh + 2 * i;
  *reinterpret_cast<uint32_t*>(b.ring + kbase + off) = pack_bf16x2(kr0, kr1);
  *reinterpret_cast<uint32_t*>(b.ring + vbase + off) = pack_bf16x2(v0, v1);
}

cudaError_t launch_rope_ring(const Dims& D, const Buffers& b, int layer, cudaStream_t s) {
  { cudaError_t e_ = launch_k(k_rope_ring, dim3(dim3(D.B, D.H)), dim3((D.Dh / 2 + 31) / 32 * 32), 0, s, 1, D, b, layer); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// ---- greedy heads ----------------------------------------------------------------------
// Argmax over fp32 logits: the lowest index holding the maximum; NaN is never chosen
// and raises PP_S_NAN.  The comparison is order independent, so any reduction tree
// gives the same index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ int block_argmax(const float* __restrict__ lg, int n, uint32_t* status) {
  __shared__ float sv[32];
  __shared__ int si[32];
  __shared__ int nan_seen;
  if (threadIdx.x == 0) nan_seen = 0;
  __syncthreads();
  float bv = -INFINITY;
  int bi = 0x7FFFFFFF;
  bool nan = false;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const float v = lg[i];
    if (isnan(v)) { nan = true; continue; }
    if (better(v, i, bv, bi)) { bv = v; bi = i; }
  }
  if (nan) nan_seen = 1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
      if (better(sv[w], si[w], sv[0], si[0])) { sv[0] = sv[w]; si[0] = si[w]; }
    if (nan_seen) atomicOr(status, PP_S_NAN);
    if (si[0] == 0x7FFFFFFF) si[0] = 0;
  }
  __syncthreads();
  const int r = si[0];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(1024) k_text_argmax(Dims D, Buffers b) {
  extern __shared__ float s_row[];
  pdl_wait_and_trigger();
  const int s = blockIdx.x;
  if (!b.live[s]) {
    if (threadIdx.x == 0) { b.out_col[s * kRows] = -1; b.tok[s] = 0; }
    return;
  }
  const float* lg = b.logits + (size_t)s * D.logits_ld;
  const SampleParams& sp = b.samp[s];
  const bool forced = b.in_fmask[s * kRows] != 0;
  const int pos = b.pos[s];
  int am;
  if (D.samp_text && sp.t_temp > 0.f && !forced) {
    const uint64_t seed = ((uint64_t)sp.seed_hi << 32) | sp.seed_lo;
    const int nh = sp.penalty != 1.f ? min(sp.window, b.hist_len[s]) : 0;
    am = block_sample<1024>(lg, D.Vt, sp.t_temp, sp.t_top_k, sp.t_top_p, sp.penalty,
                            b.hist + (size_t)s * kHist, nh, pos, samp::uniform(seed, pos, 0),
                            b.status, s_row);
  } else {
    am = block_argmax(lg, D.Vt, b.status);
  }
  if (threadIdx.x == 0) {
    int t = am;
    if (forced) {
      t = b.in_forced[s * kRows];
      if (t < 0 || t > D.Vt) { atomicOr(b.status, PP_S_INDEX); t = D.Vt; }
    }
    b.out_col[s * kRows] = t;
    b.tok[s] = t;
    b.hist[(size_t)s * kHist + (pos & (kHist - 1))] = t;   // the repetition-penalty window
    b.hist_len[s] = min(b.hist_len[s] + 1, kHist);
  }
}

cudaError_t launch_text_argmax(const Dims& D, const Buffers& b, cudaStream_t s) {
  const size_t smem = D.samp_text ? (size_t)D.Vt * sizeof(float) : 0;
  { cudaError_t e_ = launch_k(k_text_argmax, dim3(D.B), dim3(1024), smem, s, 1, D, b); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// Step k of the depformer decides row k+1: agent rows 1..8 are greedy unless forced,
// user rows 9..16 take this frame's user codes.
__global__ void __launch_bounds__(1024) k_dep_argmax(Dims D, Buffers b, int step) {
  extern __shared__ float s_row[];
  pdl_wait_and_trigger();
  const int s = blockIdx.x, row = step + 1;
  if (!b.live[s]) {
    if (threadIdx.x == 0) {
      b.out_col[s * kRows + row] = -1;
      b.tok[s] = 0;
      if (D.dep_batched && step == D.dep_steps - 1)
        for (int c = 0; c < kDepBatch; ++c) b.tokb[(size_t)c * D.B + s] = 0;
    }
    return;
  }
  int t = 0;
  if (row <= PP_AGENT_ROWS && !b.in_fmask[s * kRows + row]) {
    const float* lg = b.logits + (size_t)s * D.logits_ld + D.Vt + (size_t)step * D.Va;
    const SampleParams& sp = b.samp[s];
    if (D.samp_audio && sp.a_temp > 0.f) {
      const uint64_t seed = ((uint64_t)sp.seed_hi << 32) | sp.seed_lo;
      const int pos = b.pos[s];
      t = block_sample<1024>(lg, D.Va, sp.a_temp, sp.a_top_k, sp.a_top_p, 1.f, nullptr, 0, -1,
                             samp::uniform(seed, pos, row), b.status, s_row);
    } else {
      t = block_argmax(lg, D.Va, b.status);
    }
  }
  if (threadIdx.x == 0) {
    if (row <= PP_AGENT_ROWS) {
      if (b.in_fmask[s * kRows + row]) t = b.in_forced[s * kRows + row];
    } else {
      t = b.in_user[s * PP_USER_ROWS + row - 1 - PP_AGENT_ROWS];
    }
    if (t < 0 || t > D.Va) { atomicOr(b.status, PP_S_INDEX); t = D.Va; }
    b.out_col[s * kRows + row] = t;
    b.tok[s] = t;
    if (D.dep_batched && step == D.dep_steps - 1) {
      // the tokens of the batched steps: row 8 (just decided), then the user codes of
      // rows 9..15
      b.tokb[s] = t;
      for (int c = 1; c < kDepBatch; ++c) {
        int u = b.in_user[s * PP_USER_ROWS + c - 1];
        if (u < 0 || u > D.Va) u = D.Va;   // flagged where the user rows are written
        b.tokb[(size_t)c * D.B + s] = u;
      }
    }
  }
}

cudaError_t launch_dep_argmax(const Dims& D, const Buffers& b, int step, cudaStream_t s) {
  const size_t smem = D.samp_audio ? (size_t)D.Va * sizeof(float) : 0;
  { cudaError_t e_ = launch_k(k_dep_argmax, dim3(D.B), dim3(1024), smem, s, 1, D, b, step); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

// Rows of logits sampled independently with the caller's uniforms (pp_sample).
__global__ void __launch_bounds__(1024)
    k_sample_rows(const float* __restrict__ logits, int64_t ld, int n, float temperature,
                  int top_k, float top_p, float penalty, const int32_t* __restrict__ hist,
                  int hist_ld, const int32_t* __restrict__ hist_n,
                  const float* __restrict__ uniforms, int32_t* __restrict__ tokens,
                  uint32_t* status) {
  extern __shared__ float s_row[];
  pdl_wait_and_trigger();
  const int r = blockIdx.x;
  const int nh = hist ? max(0, min(hist_n[r], hist_ld)) : 0;
  const int t = block_sample<1024>(logits + (size_t)r * ld, n, temperature, top_k, top_p, penalty,
                                   hist ? hist + (size_t)r * hist_ld : nullptr, nh, -1,
                                   uniforms[r], status, s_row);
  if (threadIdx.x == 0) tokens[r] = t;
}

cudaError_t launch_sample_rows(const float* logits, int64_t ld, int rows, int n, float temperature,
                               int top_k, float top_p, float penalty, const int32_t* hist,
                               int hist_ld, const int32_t* hist_n, const float* uniforms,
                               int32_t* tokens, uint32_t* status, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(k_sample_rows, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSampleSmemMax);
  if (e != cudaSuccess) return e;
  e = launch_k(k_sample_rows, dim3(rows), dim3(1024), (size_t)n * sizeof(float), s, 1, logits, ld,
               n, temperature, top_k, top_p, penalty, hist, hist_ld, hist_n, uniforms, tokens,
               status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t sample_setup(const Dims& D) {
  cudaError_t e = cudaSuccess;
  if (D.samp_text)
    e = cudaFuncSetAttribute(k_text_argmax, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             D.Vt * (int)sizeof(float));
  if (e == cudaSuccess && D.samp_audio)
    e = cudaFuncSetAttribute(k_dep_argmax, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             D.Va * (int)sizeof(float));
  return e;
}

// ---- depformer step attention ------------------------------------------------------------
// One CTA per slot, one warp per head.  Appends this step's k, v (fp32) to the frame's
// cache and attends causally over steps 0..step (no positional encoding); the cache is
// indexed by step, so a new frame overwrites it from step 0 (reset each frame).
template <int E>  // head dim / 32
__global__ void __launch_bounds__(kDepAttnMaxThreads(32 * E))
k_dep_attn(Dims D, Buffers b, int step, int layer, bool op) {
  pdl_wait_and_trigger();
  pdl_trigger();   // small kernel: the next contraction may set up and prefetch meanwhile
  const int s = blockIdx.x, h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (h >= D.Hd) return;
  float* out = b.dout + (size_t)s * D.dd + h * D.Dhd;
  if (!b.live[s]) {
    for (int e = 0; e < E; ++e) {
      out[lane + 32 * e] = 0.f;
      if (op) op_store(b.op_do, D.dd, D.Bp, s, h * D.Dhd + lane + 32 * e, 0.f);
    }
    return;
  }
  const float* row = b.dqkv + (size_t)s * 3 * D.dd + h * D.Dhd;
  float* cache = b.dkv + ((size_t)s * D.Ld + layer) * D.nq * 2 * D.dd;
  // every load first (this step's q, k, v and the frame's earlier steps, all independent),
  // then the cache append: a store between them would order the later loads after it
  float q[E], kk[E], vv[E], kc[16][E], vc[16][E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    q[e] = row[lane + 32 * e];
    kk[e] = row[D.dd + lane + 32 * e];
    vv[e] = row[2 * D.dd + lane + 32 * e];
  }
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    if (t >= step) break;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      kc[t][e] = cache[(size_t)t * 2 * D.dd + h * D.Dhd + lane + 32 * e];
      vc[t][e] = cache[(size_t)t * 2 * D.dd + D.dd + h * D.Dhd + lane + 32 * e];
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    cache[(size_t)step * 2 * D.dd + h * D.Dhd + lane + 32 * e] = kk[e];
    cache[(size_t)step * 2 * D.dd + D.dd + h * D.Dhd + lane + 32 * e] = vv[e];
  }
  const float scale = 1.0f / sqrtf((float)D.Dhd);
  float sc[16];
  float m = -INFINITY;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    if (t > step) break;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) dot = fmaf(q[e], (t == step) ? kk[e] : kc[t][e], dot);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    sc[t] = dot * scale;
    m = fmaxf(m, sc[t]);
  }
  float l = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    if (t > step) break;
    const float p = expf(sc[t] - m);
    l += p;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(p, (t == step) ? vv[e] : vc[t][e], acc[e]);
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float v = acc[e] / l;
    out[lane + 32 * e] = v;
    if (op) op_store(b.op_do, D.dd, D.Bp, s, h * D.Dhd + lane + 32 * e, v);
  }
}

cudaError_t launch_dep_attn(const Dims& D, const Buffers& b, int step, int layer, bool op,
                            cudaStream_t s) {
  const int threads = D.Hd * 32;
  switch (D.Dhd) {
    case 32: { cudaError_t e_ = launch_k(k_dep_attn<1>, dim3(D.B), dim3(threads), 0, s, 1, D, b, step, layer, op); if (e_ != cudaSuccess) return e_; } break;
    case 64: { cudaError_t e_ = launch_k(k_dep_attn<2>, dim3(D.B), dim3(threads), 0, s, 1, D, b, step, layer, op); if (e_ != cudaSuccess) return e_; } break;
    case 128: { cudaError_t e_ = launch_k(k_dep_attn<4>, dim3(D.B), dim3(threads), 0, s, 1, D, b, step, layer, op); if (e_ != cudaSuccess) return e_; } break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ---- the batched user steps -------------------------------------------------------------
// Steps 8..15 of a frame take known tokens (row 8, then the user codes), so they run as one
// pass.  One CTA per (slot, step 8 + c), one warp per head: step 8 + c attends over steps
// 0..8+c with the same arithmetic, in the same order, as the one-step kernel above.  The
// keys and values of steps 0..7 come from the frame's cache, those of steps 8..8+c
// straight from this pass's qkv rows.  Nothing reads cache rows 8..15 within the frame, and
// the next frame overwrites the cache from step 0, so this pass appends nothing.
template <int E>  // head dim / 32
__global__ void __launch_bounds__(kDepAttnMaxThreads(32 * E))
k_dep_attn_b(Dims D, Buffers b, int layer) {
  pdl_wait_and_trigger();
  pdl_trigger();   // small kernel: the next contraction may set up and prefetch meanwhile
  const int s = blockIdx.x, c = blockIdx.y, h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (h >= D.Hd) return;
  const int k0 = D.nq - kDepBatch, step = k0 + c;
  uint16_t* op = b.op_dob + (size_t)c * 2 * D.Bp * D.dd;
  float* out = b.dout_b + ((size_t)c * D.B + s) * D.dd;
  if (!b.live[s]) {
    for (int e = 0; e < E; ++e) {
      const int i = h * D.Dhd + lane + 32 * e;
      out[i] = 0.f;
      op_store(op, D.dd, D.Bp, s, i, 0.f);
    }
    return;
  }
  const float* cache = b.dkv + ((size_t)s * D.Ld + layer) * D.nq * 2 * D.dd;
  // this lane's dims of this head: steps 0..k0-1 from the cache, k0..step and the query
  // from this pass's qkv rows, all loaded at once
  float kc[16][E], vc[16][E], q[E];
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    if (t >= k0) break;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      kc[t][e] = cache[(size_t)t * 2 * D.dd + h * D.Dhd + lane + 32 * e];
      vc[t][e] = cache[(size_t)t * 2 * D.dd + D.dd + h * D.Dhd + lane + 32 * e];
    }
  }
#pragma unroll
  for (int c2 = 0; c2 < kDepBatch; ++c2) {
    if (c2 > c) break;
    const float* row = b.dqkv_b + ((size_t)c2 * D.B + s) * 3 * D.dd + h * D.Dhd;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      kc[16 - kDepBatch + c2][e] = row[D.dd + lane + 32 * e];
      vc[16 - kDepBatch + c2][e] = row[2 * D.dd + lane + 32 * e];
      if (c2 == c) q[e] = row[lane + 32 * e];
    }
  }
  const float scale = 1.0f / sqrtf((float)D.Dhd);
  float sc[16];
  float m = -INFINITY;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    if (t > step) break;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) dot = fmaf(q[e], kc[t][e], dot);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    sc[t] = dot * scale;
    m = fmaxf(m, sc[t]);
  }
  float l = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    if (t > step) break;
    const float p = expf(sc[t] - m);
    l += p;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(p, vc[t][e], acc[e]);
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float v = acc[e] / l;
    const int i = h * D.Dhd + lane + 32 * e;
    out[i] = v;
    op_store(op, D.dd, D.Bp, s, i, v);
  }
}

cudaError_t launch_dep_attn_batch(const Dims& D, const Buffers& b, int layer, cudaStream_t s) {
  const int threads = D.Hd * 32;
  const dim3 grid(D.B, kDepBatch);
  switch (D.Dhd) {
    case 32: return launch_k(k_dep_attn_b<1>, grid, dim3(threads), 0, s, 1, D, b, layer);
    case 64: return launch_k(k_dep_attn_b<2>, grid, dim3(threads), 0, s, 1, D, b, layer);
    case 128: return launch_k(k_dep_attn_b<4>, grid, dim3(threads), 0, s, 1, D, b, layer);
    default: return cudaErrorInvalidValue;
  }
}

// ---- depformer step input from the all-steps in-projection ------------------------------
// One CTA per slot and step chunk: y = P_k z (this tick's contraction of all 16 steps'
// in-projections, pz[B][nq * dd], scaled by the final norm) + D_k[tok_k] (bf16 table row),
// the first layer's normalised operand (alpha * y as bf16 hi/lo) and the slot's sum of y^2
// (one partial: dims in thread order, then a fixed-order block sum).  Chunk c (grid.y)
// is step k0 + c, with its token table tok + c * B and output strides as given.
__global__ void __launch_bounds__(256) k_dep_in(Dims D, Buffers b, int k0, const int32_t* tok,
                                                const uint16_t* emb, long long emb_chunk,
                                                float* y, long long y_chunk, uint16_t* op,
                                                long long op_chunk, float* ssq) {
  __shared__ float sh[9];
  pdl_wait_and_trigger();
  pdl_trigger();   // small kernel: the next contraction may set up and prefetch meanwhile
  const int s = blockIdx.x, c = blockIdx.y, k = k0 + c;
  const int t = tok[(size_t)c * D.B + s];
  const float* pz = b.pz + (size_t)s * D.nq * D.dd + (size_t)k * D.dd;
  const uint16_t* e = emb + c * emb_chunk + (size_t)t * D.dd;
  float* yo = y + c * y_chunk + (size_t)s * D.dd;
  uint16_t* opc = op + c * op_chunk;
  float ss = 0.f;
  for (int i = threadIdx.x * 4; i < D.dd; i += 256 * 4) {
    const float4 p = *reinterpret_cast<const float4*>(pz + i);
    const uint2 w = *reinterpret_cast<const uint2*>(e + i);
    const float v[4] = {p.x + __uint_as_float(w.x << 16), p.y + __uint_as_float(w.x & 0xFFFF0000u),
                        p.z + __uint_as_float(w.y << 16), p.w + __uint_as_float(w.y & 0xFFFF0000u)};
    *reinterpret_cast<float4*>(yo + i) = make_float4(v[0], v[1], v[2], v[3]);
    const float4 al = *reinterpret_cast<const float4*>(b.dep_attn_alpha + i);
    const float av[4] = {al.x, al.y, al.z, al.w};
    uint16_t hi[4], lo[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      bf16_split(av[q] * v[q], hi[q], lo[q]);
      ss += v[q] * v[q];
    }
    *reinterpret_cast<uint2*>(opc + (size_t)s * D.dd + i) =
        make_uint2((uint32_t)hi[0] | ((uint32_t)hi[1] << 16), (uint32_t)hi[2] | ((uint32_t)hi[3] << 16));
    *reinterpret_cast<uint2*>(opc + (size_t)(D.Bp + s) * D.dd + i) =
        make_uint2((uint32_t)lo[0] | ((uint32_t)lo[1] << 16), (uint32_t)lo[2] | ((uint32_t)lo[3] << 16));
  }
  ss = block_sum<256>(ss, sh);
  if (threadIdx.x == 0) ssq[(size_t)c * D.B + s] = ss;
}

cudaError_t launch_dep_in(const Dims& D, const Buffers& b, int k0, int chunks, const int32_t* tok,
                          const uint16_t* emb, long long emb_chunk, float* y, long long y_chunk,
                          uint16_t* op, long long op_chunk, cudaStream_t s) {
  if (D.dd % 4) return cudaErrorInvalidValue;
  return launch_k(k_dep_in, dim3(D.B, chunks), dim3(256), 0, s, 1, D, b, k0, tok, emb, emb_chunk,
                  y, y_chunk, op, op_chunk, b.ssq);
}

// Rows 9..16 straight from this frame's user codes (when depformer steps 8..15, whose
// only other output is their logits, are not run).
__global__ void k_user_rows(Dims D, Buffers b) {
  pdl_wait_and_trigger();
  const int s = blockIdx.x, r = threadIdx.x;
  if (r >= PP_USER_ROWS) return;
  const int row = PP_AGENT_ROWS + 1 + r;
  if (!b.live[s]) {
    b.out_col[s * kRows + row] = -1;
    return;
  }
  int t = b.in_user[s * PP_USER_ROWS + r];
  if (t < 0 || t > D.Va) { atomicOr(b.status, PP_S_INDEX); t = D.Va; }
  b.out_col[s * kRows + row] = t;
}

cudaError_t launch_user_rows(const Dims& D, const Buffers& b, cudaStream_t s) {
  return launch_k(k_user_rows, dim3(D.B), dim3(32), 0, s, 1, D, b);
}

// ---- end of tick -----------------------------------------------------------------------
__global__ void k_finish(Dims D, Buffers b) {
  pdl_wait_and_trigger();
  const int s = blockIdx.x, r = threadIdx.x;
  if (!b.live[s]) {
    if (r < kRows) b.out_col[s * kRows + r] = -1;
    return;
  }
  if (r == 0) b.pos[s] += 1;
}

cudaError_t launch_finish(const Dims& D, const Buffers& b, cudaStream_t s) {
  { cudaError_t e_ = launch_k(k_finish, dim3(D.B), dim3(32), 0, s, 1, D, b); if (e_ != cudaSuccess) return e_; }
  return cudaGetLastError();
}

}  // namespace pp
