// k_umma.cu - the tick's weight contractions on the 5th-generation tensor cores.
//
//   Y[b, m] (op)= sum_k W[m, k] x[b, k]      for every slot b and output row m
//
// Swap-AB: the bf16 weight matrix is the MMA's A operand (M = 128 output rows per
// tile), the batch is its N dimension.  Activations are fed as two bf16 rows per slot,
// hi = bf16(x) and lo = bf16(x - hi), so that x is carried to ~16 significant bits and
// the result equals an fp32-activation product to within fp32 accumulation rounding;
// the epilogue adds the hi and lo accumulator columns.  The contraction streams each
// weight byte once, so the extra N columns cost tensor-core time only, which a
// weight-streaming kernel has to spare.
//
// One CTA = one (M-tile, K-split) unit, 4 warps, two CTAs per SM; the splits of a tile
// are one cluster:
//   warp 0 lane 0  TMA producer: weight tile (one 128-row box; gate/up pairs: two
//                  64-row boxes) + activation tile per 64-wide k-block into a ring of
//                  shared-memory stages (128B swizzle);
//   warp 1 lane 0  MMA issuer: 4 x tcgen05.mma (K = 16 each) per k-block into a TMEM
//                  accumulator [128 lanes x N columns], tcgen05.commit frees the stage;
//   all 4 warps    epilogue: tcgen05.ld of their 32 TMEM lanes, hi + lo, then either
//                  the final epilogue (one split) or, when the K range is split, a
//                  reduction across the thread-block cluster formed by the tile's
//                  splits: partials meet in distributed shared memory and each CTA
//                  adds them in split order for a slice of the tile's rows, then
//                  arrives at the cluster barrier and finishes its slice before it
//                  waits there (its peers may still be reading its partial).  The split
//                  count depends only on the matrix shape and the SM count, never on
//                  the batch, so a session's bits do not depend on the other sessions.
// Every mbarrier wait is bounded; on expiry the kernel raises PP_S_TIMEOUT, drains
// its own copies (bounded), frees its TMEM and returns.
#include <cooperative_groups.h>
#include <cuda.h>
#include <math.h>

#include "pp_async.cuh"
#include "pp_tcgen05.cuh"
#include "pp_internal.cuh"

namespace pp {

namespace {

constexpr int kBK = 64;              // k elements per block (128 bytes of bf16)

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

namespace cg = cooperative_groups;

// The value the epilogue adds to the contraction: 0 (EPI_STORE), the residual (EPI_ADD)
// or the token embedding row (EPI_EMB).
__device__ __forceinline__ float epi_extra(const UmmaArgs& a, int b, int m) {
  if (a.epi == EPI_ADD) return a.Y[(size_t)b * a.ldy + m];
  return bf16_to_f32(a.emb[(size_t)a.tok[b] * a.M + m]);
}

__device__ __forceinline__ void epi_store(const UmmaArgs& a, int b, int m, float v) {
  float* y = a.Y + (size_t)b * a.ldy + m;
  if (a.epi == EPI_STORE) {
    *y = v;
  } else if (a.epi == EPI_ADD) {
    *y = v + *y;
  } else {  // EPI_EMB
    *y = v + bf16_to_f32(a.emb[(size_t)a.tok[b] * a.M + m]);
  }
}

// N: MMA columns (2 x padded slots, hi and lo); H: 128-row halves of the weight tile.
// H = 1: 4 warps, two CTAs per SM; H = 2: 8 warps, one CTA per SM, a 256-row tile whose
// two halves share every activation tile (half the activation bytes per weight byte).
// Order-preserving 64-bit key of a finite logit at a row: a larger value wins, then the
// lower row (the greedy rule); -0 counts as +0.  Any reduction order gives the same max.
// The high word (greedy_bits) is never 0 for a non-NaN value, infinities included.
__device__ __forceinline__ uint32_t greedy_bits(float v) {
  if (v == 0.f) v = 0.f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long greedy_key(float v, int row) {
  return ((unsigned long long)greedy_bits(v) << 32) |
         (unsigned long long)(0xFFFFFFFFu - (uint32_t)row);
}

// EPI_ROPE for 4 consecutive rows m..m+3 of open slot s (two RoPE pairs of one head; t:
// cos, sin of both pairs; widx: the slot's ring row): the query (scaled) to q and q_op,
// the key (rotated) and value to the ring.
__device__ __forceinline__ void rope_store(const RopeArgs& r, int s, int m, const float* y,
                                           float4 t, int widx) {
  const int sec = m / r.d, w = m - sec * r.d, h = w / r.Dh, e = w - h * r.Dh;
  const size_t blk = (size_t)r.W * r.Dh;
  const size_t at = (size_t)widx * r.Dh + e;
  uint16_t* ring = r.ring + (size_t)s * 2 * r.H * blk;
  if (sec == 2) {
    *reinterpret_cast<uint2*>(ring + (size_t)(r.H + h) * blk + at) =
        make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
    return;
  }
  float o[4] = {y[0] * t.x - y[1] * t.y, y[0] * t.y + y[1] * t.x,
                y[2] * t.z - y[3] * t.w, y[2] * t.w + y[3] * t.z};
  if (sec == 1) {
    *reinterpret_cast<uint2*>(ring + (size_t)h * blk + at) =
        make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
    return;
  }
  const float qs = 1.4426950408889634f / sqrtf((float)r.Dh);
  uint16_t hi[4], lo[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    o[c] *= qs;
    bf16_split(o[c], hi[c], lo[c]);
  }
  *reinterpret_cast<float4*>(r.q + (size_t)s * r.d + w) = make_float4(o[0], o[1], o[2], o[3]);
  uint16_t* qo = r.q_op + (size_t)(s * r.H + h) * 2 * r.Dh + e;
  *reinterpret_cast<uint2*>(qo) = make_uint2((uint32_t)hi[0] | ((uint32_t)hi[1] << 16),
                                             (uint32_t)hi[2] | ((uint32_t)hi[3] << 16));
  *reinterpret_cast<uint2*>(qo + r.Dh) = make_uint2((uint32_t)lo[0] | ((uint32_t)lo[1] << 16),
                                                    (uint32_t)lo[2] | ((uint32_t)lo[3] << 16));
}

// The fused greedy decision of a head contraction: each CTA folds its per-slot keys
// (best[b]) into the launch's global key of each slot with an atomic max, and its NaN
// flag (flags[0]) into a global flag; the last CTA to finish reads the B keys, resets them
// for the next launch, and takes each slot's decision (forced token, greedy token, or
// user code), as the decision kernels of the sampling-capable tick do for greedy slots.
__device__ void decide_tail(const UmmaArgs& a, unsigned long long* best, unsigned* flags, int B) {
  const DecideArgs& d = a.dec;
  const int units = gridDim.x;
  __syncthreads();
  if (threadIdx.x < B && best[threadIdx.x]) atomicMax(d.key + threadIdx.x, best[threadIdx.x]);
  if (threadIdx.x == 0 && flags[0]) atomicOr(d.nan, 1u);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    flags[1] = (atomicAdd(d.ticket, 1u) == (unsigned)units - 1u) ? 1u : 0u;
  }
  __syncthreads();
  if (!flags[1]) return;
  __threadfence();
  if (threadIdx.x < B) {
    best[threadIdx.x] = __ldcg(d.key + threadIdx.x);
    d.key[threadIdx.x] = 0ull;   // ready for the next launch
  }
  if (threadIdx.x == 0) {
    flags[0] = __ldcg(d.nan);
    *d.nan = 0u;
  }
  __syncthreads();
  if (threadIdx.x < B) {
    const int s = threadIdx.x;
    const unsigned long long k = best[s];
    const int am = k ? (int)(0xFFFFFFFFu - (uint32_t)k) : 0;   // all NaN: token 0
    const bool nan = flags[0] != 0u;
    if (d.kind == 1) {   // text row 0
      if (!d.live[s]) {
        d.out_col[s * kRows] = -1;
        d.tok[s] = 0;
      } else {
        int t = am;
        if (d.fmask[s * kRows]) {
          t = d.forced[s * kRows];
          if (t < 0 || t > d.V) { atomicOr(a.status, PP_S_INDEX); t = d.V; }
        } else if (nan) {
          atomicOr(a.status, PP_S_NAN);
        }
        d.out_col[s * kRows] = t;
        d.tok[s] = t;
        const int pos = d.pos[s];
        d.hist[(size_t)s * d.hist_ld + (pos & (d.hist_ld - 1))] = t;
        d.hist_len[s] = min(d.hist_len[s] + 1, d.hist_ld);
      }
    } else {             // depformer step `step` decides row step + 1
      const int row = d.step + 1;
      if (!d.live[s]) {
        d.out_col[s * kRows + row] = -1;
        d.tok[s] = 0;
        if (d.tokb)
          for (int c = 0; c < kDepBatch; ++c) d.tok_b[(size_t)c * B + s] = 0;
      } else {
        int t;
        if (row <= PP_AGENT_ROWS) {
          if (d.fmask[s * kRows + row]) {
            t = d.forced[s * kRows + row];
          } else {
            t = am;
            if (nan) atomicOr(a.status, PP_S_NAN);
          }
        } else {
          t = d.user[s * PP_USER_ROWS + row - 1 - PP_AGENT_ROWS];
        }
        if (t < 0 || t > d.V) { atomicOr(a.status, PP_S_INDEX); t = d.V; }
        d.out_col[s * kRows + row] = t;
        d.tok[s] = t;
        if (d.tokb) {
          d.tok_b[s] = t;
          for (int c = 1; c < kDepBatch; ++c) {
            int u = d.user[s * PP_USER_ROWS + c - 1];
            if (u < 0 || u > d.V) u = d.V;
            d.tok_b[(size_t)c * B + s] = u;
          }
        }
      }
    }
  }
  if (threadIdx.x == 0) *d.ticket = 0u;   // ready for the next launch
}

template <int N, int H>
struct Cfg {
  static constexpr int kRows = 128 * H;                  // weight rows per tile
  static constexpr int kPairs = 64 * H;                  // gate/up pairs per tile
  static constexpr int kThreads = 128 * H;
  static constexpr int kABytes = kRows * kBK * 2;        // weight tile (H x 16 KB)
  static constexpr int kBBytes = N * kBK * 2;            // activation tile
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBudget = (H == 1 ? 96 : 192) * 1024;
  static constexpr int kStages = kBudget / kStageBytes < 8 ? kBudget / kStageBytes : 8;
  static constexpr int kCols = H * N;                    // accumulator columns (TMEM)
  static constexpr int kTmemCols = kCols <= 32 ? 32 : (kCols <= 64 ? 64 : (kCols <= 128 ? 128 : (kCols <= 256 ? 256 : 512)));
  static constexpr int kSmem = kStages * kStageBytes + 1024 /*align*/ + 512 /*barriers, 1/rms*/;
  // the split-K epilogue reuses the idle stages: partial + y^2 [2][N/2][kPR] floats
  static constexpr int kPR = kRows + 4;                  // row stride of a parked partial
  // fused greedy decision: [64] keys and 2 flags after the partials
  static constexpr int kKeyOff = ((2 * (N / 2) * kPR * 4) + 1023) / 1024 * 1024;
  static_assert(kKeyOff + 64 * 8 + 16 <= kStages * kStageBytes, "decision keys");
  static_assert((N / 2) * (kRows + 1) * 4 <= kKeyOff, "slot-major logits of a head tile");
  // single split: SiLU exchange [kPairs][N/2] and y^2 [kRows][N/2 + 1] in the stages
  static_assert(kRows * (N / 2 + 1) * 4 <= kStages * kStageBytes, "y^2 area");
  static_assert(kStages >= 2, "pipeline depth");
};

template <int N, int H>
__global__ void __launch_bounds__(128 * H, H == 1 ? 2 : 1)
    k_umma(const UmmaArgs a_in, const __grid_constant__ CUtensorMap mapA,
           const __grid_constant__ CUtensorMap mapB) {
  using C = Cfg<N, H>;
  // column chunk c: this chunk's operand rows, weights and outputs
  const int chunk = blockIdx.y;
  UmmaArgs a = a_in;
  if (chunk) {
    a.row0 += chunk * a.a_chunk_rows;
    if (a.Y) a.Y += chunk * a.y_chunk;
    if (a.norm_op) a.norm_op += chunk * a.op_chunk;
    if (a.op_out) a.op_out += chunk * a.op_chunk;
    if (a.ssq_out) a.ssq_out += chunk * a.ssq_out_chunk;
    if (a.ssq_in) a.ssq_in += chunk * a.ssq_in_chunk;
    if (a.emb) a.emb += chunk * a.emb_chunk;
    if (a.tok) a.tok += chunk * a.tok_chunk;
  }
  const int brow = chunk * a.b_chunk_rows;   // first operand row of this chunk
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  // bars[0..S) full, bars[S..2S) empty, bars[2S] done; then the TMEM address and flags
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* s_rstd = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes + 256);  // [B]
  const bool norm_in = a.ssq_in != nullptr || a.rstd_in != nullptr;
  const bool norm_out = a.norm_alpha != nullptr;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x / a.splits, sp = blockIdx.x % a.splits;
  const int kb0 = (int)(((long long)sp * a.kblocks) / a.splits);
  const int kb1 = (int)(((long long)(sp + 1) * a.kblocks) / a.splits);
  const int nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[C::kStages + s]), 1);
    }
    mbar_init(smem_u32(&bars[2 * C::kStages]), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(C::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  if (a.early_trigger) pdl_trigger();

  // rows of the weight boxes of this tile: the tile's kRows rows (boxes of 128 rows),
  // or its kPairs gate rows then the matching up rows (boxes of kPairs rows)
  int rowA0, rowA1;
  if (a.pair_rows) {
    rowA0 = a.row0 + mt * C::kPairs;
    rowA1 = a.row0 + a.pair_rows + mt * C::kPairs;
  } else {
    rowA0 = a.row0 + mt * C::kRows;
    rowA1 = rowA0 + 128;
  }

  if (warp == 0 && lane == 0) {
    // ---- TMA producer ------------------------------------------------------------------
    // The weights do not depend on the previous kernel: the first stages' weight tiles
    // are requested before waiting for it (programmatic dependent launch), the
    // activation tiles after.
    int32_t armed, kinds;
    read_withhold(a.test_ctl, armed, kinds);   // used after the dependency wait
    const int pre = nkb < C::kStages ? nkb : C::kStages;
    // weight tile of one k-block, [kRows][64] swizzled: H boxes of 128 rows, or (gate/up
    // pairs) a box of the gate rows and a box of the up rows, kPairs rows each
    auto load_a = [&](uint8_t* sa, int kx, uint32_t full) {
      tma_load_2d(smem_u32(sa), &mapA, kx, rowA0, full);
      if (a.pair_rows || H == 2) tma_load_2d(smem_u32(sa + C::kABytes / 2), &mapA, kx, rowA1, full);
    };
    for (int i = 0; i < pre; ++i) {
      uint8_t* sa = smem + i * C::kStageBytes;
      const uint32_t full = smem_u32(&bars[i]);
      mbar_expect_tx(full, C::kStageBytes);
      load_a(sa, (kb0 + i) * kBK, full);
    }
    pdl_wait_and_trigger();
    int issued = 0;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % C::kStages;
      if (i >= C::kStages &&
          !mbar_wait(smem_u32(&bars[C::kStages + s]), ((i / C::kStages) - 1) & 1, a.test_ctl)) {
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      uint8_t* sa = smem + s * C::kStageBytes;
      uint8_t* sb = sa + C::kABytes;
      const uint32_t full = smem_u32(&bars[s]);
      const int kx = (kb0 + i) * kBK;
      if (i >= pre) {
        mbar_expect_tx(full, C::kStageBytes);
        load_a(sa, kx, full);
      }
      // a failure-detection test may have this producer withhold the first activation
      // tile: its stage never completes and the MMA issuer's bounded wait runs out
      if (!(i == 0 && take_withhold(a.test_ctl, armed, kinds, PP_TEST_UMMA)))
        tma_load_2d(smem_u32(sb), &mapB, kx, brow, full);
      ++issued;
    }
    if (*abort_flag) {  // drain this CTA's copies still in flight (bounded waits)
      const int inflight = issued > pre ? issued : pre;
      for (int i = 0; i < inflight; ++i)
        mbar_wait(smem_u32(&bars[i % C::kStages]), (i / C::kStages) & 1, a.test_ctl);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer --------------------------------------------------------------------
    constexpr uint32_t idesc = instr_desc(128, N);
    for (int i = 0; i < nkb; ++i) {
      const int s = i % C::kStages;
      if (!mbar_wait(smem_u32(&bars[s]), (i / C::kStages) & 1, a.test_ctl)) {
        *abort_flag = 1;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t sa = smem_u32(smem + s * C::kStageBytes);
      const uint32_t sb = sa + C::kABytes;
#pragma unroll
      for (int h = 0; h < H; ++h)
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          umma_bf16(tmem + h * N, smem_desc(sa + h * 16384 + kk * 32), smem_desc(sb + kk * 32),
                    idesc, (i > 0 || kk > 0) ? 1u : 0u);
      umma_commit(smem_u32(&bars[C::kStages + s]));
    }
    umma_commit(smem_u32(&bars[2 * C::kStages]));
  } else if (warp >= 2 && norm_in) {
    pdl_wait_and_trigger();
    // fused RMSNorm of the input: 1/rms of every slot, summed from the producer's
    // partials in slice order while the main loop runs
    for (int b = threadIdx.x - 64; b < a.B; b += C::kThreads - 64) {
      float rs;
      if (a.rstd_in) {
        rs = a.rstd_in[b];
      } else {
        float ss = 0.f;
        for (int q0 = 0; q0 < a.ssq_nparts; q0 += 16) {   // 16 loads in flight, added in order
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            v[i] = (q0 + i < a.ssq_nparts) ? a.ssq_in[(size_t)(q0 + i) * a.B + b] : 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) ss += v[i];
        }
        rs = 1.0f / sqrtf(ss / (float)a.ssq_K + a.eps);
      }
      s_rstd[b] = rs;
      if (a.rstd_out && blockIdx.x == 0) a.rstd_out[b] = rs;
    }
  }
  if (!(warp == 0 && lane == 0)) pdl_wait_and_trigger();   // (a no-op when done twice)
  __syncwarp();

  // ---- epilogue ----------------------------------------------------------------------
  const bool done = mbar_wait(smem_u32(&bars[2 * C::kStages]), 0, a.test_ctl);
  if (!done) *abort_flag = 1;
  pdl_trigger();   // main loop over: the next kernel may start launching
  __syncthreads();
  const bool ok = !*abort_flag && nkb > 0;
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  // this thread: TMEM lane r of accumulator half `half`, i.e. row tr of the tile
  const int half = warp >> 2;
  const int r = (warp & 3) * 32 + lane;
  const int tr = half * 128 + r;
  const int B = a.B, Bp = N / 2;
  // output row of this thread: tile row, or pair p (gate when `gate`, else up)
  const bool gate = (H == 1) ? (r < 64) : (half == 0);
  const int p = (H == 1) ? (r & 63) : r;
  int m;
  if (a.pair_rows) m = mt * C::kPairs + p;
  else m = mt * C::kRows + tr;
  const bool row_ok = a.pair_rows ? (m < a.pair_rows) : (m < a.M);

  float acc[N / 2];
  {
    uint32_t hi[N / 2], lo[N / 2];
    const uint32_t t = tmem + ((uint32_t)((warp & 3) * 32) << 16) + half * N;
    if (ok) {
#pragma unroll
      for (int c = 0; c < N / 2; c += 8) {
        tmem_ld8(t + c, hi + c);
        tmem_ld8(t + Bp + c, lo + c);
      }
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < N / 2; ++c) acc[c] = after_wait(hi[c]) + after_wait(lo[c]);
    } else {
#pragma unroll
      for (int c = 0; c < N / 2; ++c) acc[c] = 0.f;
    }
  }
  unsigned long long* s_best = reinterpret_cast<unsigned long long*>(smem + C::kKeyOff);
  unsigned* s_dflags = reinterpret_cast<unsigned*>(smem + C::kKeyOff + 64 * 8);
  if (a.dec.kind) {   // the stages are idle: per-slot best keys of the fused decision
    if (threadIdx.x < 64) s_best[threadIdx.x] = 0ull;
    if (threadIdx.x == 0) s_dflags[0] = 0u;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::kTmemCols));

  // ---- final epilogue, single split: straight from the accumulator registers ------------
  if (a.splits == 1) {
    if (!ok) {
      if (threadIdx.x == 0 && nkb > 0) atomicOr(a.status, PP_S_TIMEOUT);
      return;
    }
    if (norm_in) {
#pragma unroll
      for (int b = 0; b < N / 2; ++b)
        if (b < B) acc[b] *= s_rstd[b];
    }
    if (a.epi == EPI_SILU) {
      float* xch = reinterpret_cast<float*>(smem);   // stages idle now: [kPairs][Bp] up values
      if (!gate) {
#pragma unroll
        for (int b = 0; b < N / 2; ++b)
          if (b < B) xch[p * Bp + b] = acc[b];
      }
      __syncthreads();
      if (gate && row_ok) {
#pragma unroll
        for (int b = 0; b < N / 2; ++b) {
          if (b < B) {
            const float g = acc[b], u = xch[p * Bp + b];
            op_store(a.op_out, a.ld_op, a.Bp_out, b, m, g / (1.0f + expf(-g)) * u);
          }
        }
      }
      return;
    }
    if (!norm_out) {
      if (row_ok) {
#pragma unroll
        for (int b = 0; b < N / 2; ++b)
          if (b < B) epi_store(a, b, m, acc[b]);
      }
      if (a.dec.kind) {
        // the tile's logits slot-major in the idle stages, then one warp per slot: a short
        // rolled loop (this runs once per launch, from a cold instruction cache)
        constexpr int XL = C::kRows + 1;
        float* xs = reinterpret_cast<float*>(smem);   // [N/2][XL]
#pragma unroll
        for (int b = 0; b < N / 2; ++b)
          if (b < B) xs[b * XL + tr] = acc[b];
        __syncthreads();
        const int rows = min(C::kRows, a.M - mt * C::kRows);
#pragma unroll 1
        for (int b = warp; b < B; b += C::kThreads / 32) {
          uint32_t hi = 0u, row = 0u;   // rows visited in ascending order: ties keep the first
#pragma unroll 1
          for (int q = lane; q < rows; q += 32) {
            const float v = xs[b * XL + q];
            if (isnan(v)) {
              s_dflags[0] = 1u;
            } else {
              const uint32_t h = greedy_bits(v);
              if (h > hi) { hi = h; row = (uint32_t)q; }
            }
          }
          const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, hi);
          const uint32_t mr = __reduce_min_sync(0xFFFFFFFFu, hi == mx ? row : 0xFFFFFFFFu);
          if (lane == 0 && mx)
            s_best[b] = ((unsigned long long)mx << 32) |
                        (unsigned long long)(0xFFFFFFFFu - (uint32_t)(mt * C::kRows + mr));
        }
        decide_tail(a, s_best, s_dflags, B);
      }
      return;
    }
    // producer of a fused RMSNorm: y, the next operand and the tile's sums of y^2
    constexpr int PB1 = N / 2 + 1;
    float* sq = reinterpret_cast<float*>(smem);      // [kRows][PB1] y^2, stages idle now
#pragma unroll
    for (int b = 0; b < N / 2; ++b) {
      if (b < B) {
        float y = 0.f;
        if (row_ok) {
          y = acc[b] + epi_extra(a, b, m);
          a.Y[(size_t)b * a.ldy + m] = y;
          op_store(a.norm_op, a.M, Bp, b, m, a.norm_alpha[m] * y);
        }
        sq[tr * PB1 + b] = y * y;
      }
    }
    __syncthreads();
    if (threadIdx.x < B) {
      float ss = 0.f;
      for (int rr = 0; rr < C::kRows; ++rr) ss += sq[rr * PB1 + threadIdx.x];
      a.ssq_out[(size_t)mt * B + threadIdx.x] = ss;
    }
    return;
  }

  // ---- split-K across the thread-block cluster (one CTA per split of this tile) ----------
  // Each CTA parks its partial [slot][row] (row stride PR) in its own shared memory;
  // after a cluster barrier, CTA `sp` reduces a slice of the tile's rows, 4 rows aligned
  // to 4 per thread and step, reading the S partials through distributed shared memory
  // with 16-byte loads and adding them in split order 0..S-1; then it applies the
  // epilogue.  The second cluster barrier is split: a CTA arrives once it has read its
  // peers and waits (before it exits, which would free its shared memory) only after
  // its slice's stores.  Every CTA passes both barriers, also after a timeout.
  constexpr int PR = C::kPR;                 // row stride of a parked partial (16 bytes)
  float* mine = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int b = 0; b < N / 2; ++b)
    if (b < B) mine[b * PR + tr] = ok ? acc[b] : 0.f;
  // EPI_ROPE: each slot's open flag and ring row, staged once (the key area is unused)
  int* s_rope = reinterpret_cast<int*>(smem + C::kKeyOff);   // [2][64]
  if (a.epi == EPI_ROPE && threadIdx.x < B) {
    s_rope[threadIdx.x] = a.rope.live[threadIdx.x];
    s_rope[64 + threadIdx.x] = a.rope.pos[threadIdx.x] % a.rope.W;
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int S = a.splits;
  const float* peer[kMaxSplits];
#pragma unroll
  for (int q = 0; q < kMaxSplits; ++q) peer[q] = q < S ? cluster.map_shared_rank(mine, q) : mine;
  auto ld4 = [](const float* p) { return *reinterpret_cast<const float4*>(p); };
  constexpr int CH = 2;   // 4-row units per thread and step: up to 2*S 16-byte peer loads
  if (a.epi == EPI_SILU) {
    // slice of the kPairs gate/up pairs in whole 4-pair groups; unit = (slot, 4 pairs);
    // gate of pair p parked at row p, its up at row kPairs + p
    const int p0 = 4 * ((sp * (C::kPairs / 4)) / S), p1 = 4 * (((sp + 1) * (C::kPairs / 4)) / S);
    const int G = (p1 - p0) / 4;
    const int n = G * B;
    for (int u0 = threadIdx.x; u0 < n; u0 += CH * (int)blockDim.x) {
      int off[CH], mm[CH], bc[CH];
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const int u = u0 + i * (int)blockDim.x;
        const int g = u % G;
        bc[i] = u / G;
        mm[i] = (u < n) ? mt * C::kPairs + p0 + 4 * g : a.pair_rows;   // pair_rows: no unit
        off[i] = bc[i] * PR + p0 + 4 * g;
      }
      float4 gv[CH][kMaxSplits], uv[CH][kMaxSplits];
#pragma unroll
      for (int i = 0; i < CH; ++i)
#pragma unroll
        for (int q = 0; q < kMaxSplits; ++q)
          if (q < S && mm[i] < a.pair_rows) {
            gv[i][q] = ld4(peer[q] + off[i]);
            uv[i][q] = ld4(peer[q] + off[i] + C::kPairs);
          }
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        if (mm[i] >= a.pair_rows) continue;
        float g4[4] = {0.f, 0.f, 0.f, 0.f}, u4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < kMaxSplits; ++q)
          if (q < S) {
            g4[0] += gv[i][q].x; g4[1] += gv[i][q].y; g4[2] += gv[i][q].z; g4[3] += gv[i][q].w;
            u4[0] += uv[i][q].x; u4[1] += uv[i][q].y; u4[2] += uv[i][q].z; u4[3] += uv[i][q].w;
          }
        const float rs = norm_in ? s_rstd[bc[i]] : 1.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (mm[i] + c >= a.pair_rows) break;
          float g = g4[c], u = u4[c];
          if (norm_in) { g *= rs; u *= rs; }
          op_store(a.op_out, a.ld_op, a.Bp_out, bc[i], mm[i] + c, g / (1.0f + expf(-g)) * u);
        }
      }
    }
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");   // this CTA read its peers
  } else {
    // slice of the tile's kRows rows in whole 4-row groups; unit = (slot, 4 rows); units
    // run rows fastest across threads, so y and the next operand are written in rows
    const int r0 = 4 * ((sp * (C::kRows / 4)) / S), r1 = 4 * (((sp + 1) * (C::kRows / 4)) / S);
    const int G = (r1 - r0) / 4;
    const int n = G * B;
    float* sq = mine + (N / 2) * PR;  // [slot][row - r0] y^2 of this slice (fused RMSNorm)
    for (int u0 = threadIdx.x; u0 < n; u0 += CH * (int)blockDim.x) {
      int off[CH], mrow[CH], bcol[CH];
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const int u = u0 + i * (int)blockDim.x;
        const int g = u % G;
        bcol[i] = u / G;
        mrow[i] = (u < n) ? mt * C::kRows + r0 + 4 * g : a.M;   // a.M marks "no unit"
        off[i] = bcol[i] * PR + r0 + 4 * g;
      }
      float4 ex[CH], al[CH];   // residual (or embedding) and norm gains of the 4 rows
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        ex[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        al[i] = ex[i];
        if (mrow[i] < a.M) {
          if (a.epi == EPI_ADD) {
            ex[i] = ld4(a.Y + (size_t)bcol[i] * a.ldy + mrow[i]);
          } else if (a.epi == EPI_EMB) {
            const uint2 w = *reinterpret_cast<const uint2*>(
                a.emb + (size_t)a.tok[bcol[i]] * a.M + mrow[i]);
            ex[i] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                                __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
          }
          if (norm_out) al[i] = ld4(a.norm_alpha + mrow[i]);
          if (a.epi == EPI_ROPE && mrow[i] < 2 * a.rope.d) {   // q, k: cos, sin of 2 pairs
            const int w = mrow[i] % a.rope.d;
            al[i] = ld4(a.rope.cs + (size_t)bcol[i] * a.rope.Dh + w % a.rope.Dh);
          }
        }
      }
      float4 pv[CH][kMaxSplits];
#pragma unroll
      for (int i = 0; i < CH; ++i)
#pragma unroll
        for (int q = 0; q < kMaxSplits; ++q)
          if (q < S && mrow[i] < a.M) pv[i][q] = ld4(peer[q] + off[i]);
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        if (mrow[i] >= a.M) continue;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < kMaxSplits; ++q)
          if (q < S) {
            v[0] += pv[i][q].x; v[1] += pv[i][q].y; v[2] += pv[i][q].z; v[3] += pv[i][q].w;
          }
        const float rs = norm_in ? s_rstd[bcol[i]] : 1.f;
        const float exv[4] = {ex[i].x, ex[i].y, ex[i].z, ex[i].w};
        const float alv[4] = {al[i].x, al[i].y, al[i].z, al[i].w};
        float y[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float vv = v[c];
          if (norm_in) vv *= rs;
          y[c] = vv + exv[c];
        }
        if (a.epi == EPI_ROPE) {
          if (s_rope[bcol[i]]) rope_store(a.rope, bcol[i], mrow[i], y, al[i], s_rope[64 + bcol[i]]);
        } else
          *reinterpret_cast<float4*>(a.Y + (size_t)bcol[i] * a.ldy + mrow[i]) =
              make_float4(y[0], y[1], y[2], y[3]);
        if (a.dec.kind) {   // the 4 rows' best first: one shared atomic per unit
          unsigned long long k = 0ull;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (mrow[i] + c >= a.M) break;
            if (isnan(y[c])) s_dflags[0] = 1u;
            else k = max(k, greedy_key(y[c], mrow[i] + c));
          }
          if (k) atomicMax(&s_best[bcol[i]], k);
        }
        if (norm_out) {
          uint16_t hi[4], lo[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) bf16_split(alv[c] * y[c], hi[c], lo[c]);
          *reinterpret_cast<uint2*>(a.norm_op + (size_t)bcol[i] * a.M + mrow[i]) =
              make_uint2((uint32_t)hi[0] | ((uint32_t)hi[1] << 16),
                         (uint32_t)hi[2] | ((uint32_t)hi[3] << 16));
          *reinterpret_cast<uint2*>(a.norm_op + (size_t)(Bp + bcol[i]) * a.M + mrow[i]) =
              make_uint2((uint32_t)lo[0] | ((uint32_t)lo[1] << 16),
                         (uint32_t)lo[2] | ((uint32_t)lo[3] << 16));
          *reinterpret_cast<float4*>(sq + off[i] - r0) =
              make_float4(y[0] * y[0], y[1] * y[1], y[2] * y[2], y[3] * y[3]);
        }
      }
      if (norm_out) {   // units past the matrix rows add nothing
#pragma unroll
        for (int i = 0; i < CH; ++i)
          if (mrow[i] >= a.M && u0 + i * (int)blockDim.x < n)
            *reinterpret_cast<float4*>(sq + off[i] - r0) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");   // this CTA read its peers
    if (norm_out) {   // this slice's sums of y^2, in row order: one partial per CTA
      __syncthreads();
      if (threadIdx.x < B) {
        float ss = 0.f;
        for (int rr = 0; rr < r1 - r0; rr += 4) {
          const float4 w = ld4(sq + threadIdx.x * PR + rr);
          ss += w.x;
          ss += w.y;
          ss += w.z;
          ss += w.w;
        }
        a.ssq_out[((size_t)mt * S + sp) * B + threadIdx.x] = ss;
      }
    }
  }
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");   // peers done reading
  if (!ok && threadIdx.x == 0 && nkb > 0) atomicOr(a.status, PP_S_TIMEOUT);
  if (a.dec.kind) decide_tail(a, s_best, s_dflags, B);
}

}  // namespace

template <int N, int H>
static cudaError_t umma_n(const UmmaArgs& a, const CUtensorMap& mA, const CUtensorMap& mB,
                          cudaStream_t s) {
  const int grid = a.m_tiles * a.splits;
  return launch_k(k_umma<N, H>, dim3(grid, a.chunks > 1 ? a.chunks : 1), dim3(Cfg<N, H>::kThreads),
                  Cfg<N, H>::kSmem, s, a.splits, a, mA, mB);
}

template <int N>
static cudaError_t setup_n() {
  cudaError_t e = cudaFuncSetAttribute(k_umma<N, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<N, 1>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_umma<N, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<N, 2>::kSmem);
}

// Raise the dynamic shared-memory limits of the kernels for N (call before capture).
cudaError_t umma_setup(int N) {
  switch (N) {
    case 16: return setup_n<16>();
    case 32: return setup_n<32>();
    case 48: return setup_n<48>();
    case 64: return setup_n<64>();
    case 80: return setup_n<80>();
    case 96: return setup_n<96>();
    case 112: return setup_n<112>();
    case 128: return setup_n<128>();
    default: return cudaErrorInvalidValue;
  }
}

template <int N>
static cudaError_t umma_h(const UmmaArgs& a, const CUtensorMap& mA, const CUtensorMap& mB,
                          cudaStream_t s) {
  return a.halves == 2 ? umma_n<N, 2>(a, mA, mB, s) : umma_n<N, 1>(a, mA, mB, s);
}

cudaError_t launch_umma(const UmmaArgs& a, const CUtensorMap& mA, const CUtensorMap& mB,
                        cudaStream_t s) {
  if (a.halves != 1 && a.halves != 2) return cudaErrorInvalidValue;
  switch (a.N) {
    case 16: return umma_h<16>(a, mA, mB, s);
    case 32: return umma_h<32>(a, mA, mB, s);
    case 48: return umma_h<48>(a, mA, mB, s);
    case 64: return umma_h<64>(a, mA, mB, s);
    case 80: return umma_h<80>(a, mA, mB, s);
    case 96: return umma_h<96>(a, mA, mB, s);
    case 112: return umma_h<112>(a, mA, mB, s);
    case 128: return umma_h<128>(a, mA, mB, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pp
