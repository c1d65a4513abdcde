// k_attn_tc.cu - ring attention for head dim 128 on the 5th-generation tensor cores.
//
// Same work units and the same chunk partials as the CUDA-core kernel (k_attn.cu): a
// unit is (slot, head, chunk of 128 ring indices), each CTA walks a contiguous range of
// units, and the last CTA to finish a (slot, head) merges its chunks in chunk order.
// Within a unit both contractions are tcgen05 MMAs with the chunk's 128 keys (or the
// head's 128 dims) as the M = 128 rows:
//
//   S [128 keys x 16]  = K [128 keys x 128 dims] . Qop^T     Qop rows 0,1 = q_hi, q_lo
//   O [128 dims x 16]  = V^T [128 dims x 128 keys] . Pop^T   Pop rows 0,1 = p_hi, p_lo
//
// so s = S[:,0] + S[:,1] and o = O[:,0] + O[:,1] carry q and p to ~16 significant bits
// (K and V are bf16 already); the other 14 columns are never read.  K is a K-major A
// operand, V^T an MN-major one (the TMA tile of V is [keys][dims] with dims contiguous).
//
// Warp roles (384 threads, one CTA per SM):
//   warp 0 lane 0   TMA producer: K, V (two 64-dim boxes each) and the query operand of
//                   every unit into a ring of 3 shared-memory stages;
//   warp 1 lane 0   MMA issuer: S of unit v+1 is issued before O of unit v, so the
//                   softmax of one unit overlaps the next unit's scores; TMEM holds two
//                   (S, O) buffers;
//   warp 2          merge warp: per run of a (slot, head)'s chunks in this CTA, one
//                   release fence and ticket; the last CTA merges the chunk partials;
//   warps 4-7       softmax: thread t owns key t (TMEM lane t) of the chunk: chunk max
//                   and sum over the four warps, p = 2^(s - max) as bf16 hi/lo into the
//                   swizzled P operand;
//   warps 8-11      epilogue: thread t owns output dim t: the chunk partial
//                   (max, sum, o[128]) to global scratch.
// Every reduction order is fixed by ring index and hardware, never by the batch, the
// grid or timing.  Every wait is bounded; on expiry the kernel raises PP_S_TIMEOUT and
// runs to completion without further waits (results are then undefined).
#include <math.h>

#include "pp_async.cuh"
#include "pp_attn_common.cuh"
#include "pp_internal.cuh"
#include "pp_tcgen05.cuh"

namespace pp {

namespace {

using namespace attn;

constexpr int kDH = 128;
constexpr int kKStages = 2;                            // K + query ring
constexpr int kVStages = 3;                            // V ring
constexpr int kBufs = 3;                               // TMEM (S, O) and P operand buffers
// The softmax may run up to kBufs - 1 units ahead of the oldest output not yet issued;
// its wait on a V stage (ragged chunks) is only unambiguous when that stage's previous
// tile has already been consumed, i.e. when the V ring is at least kBufs deep.
static_assert(kVStages >= kBufs, "V ring shallower than the S/P buffers");
constexpr int kStash = 32;                             // chunk partials kept on chip
constexpr int kBoxBytes = kAttnChunk * 128;           // 128 rows x 64 bf16 (128 bytes)
constexpr int kKVBytes = 2 * kBoxBytes;                // two 64-dim boxes
constexpr int kQBoxBytes = 16 * 128;                   // 16 rows x 64 bf16
constexpr int kQBytes = 2 * kQBoxBytes;
constexpr int kKStageBytes = kKVBytes + kQBytes;       // K | query operand
constexpr int kVOff = kKStages * kKStageBytes;         // V ring
constexpr int kPBytes = 2 * kQBoxBytes;                // P operand: 16 rows x 128 keys
constexpr int kPOff = kVOff + kVStages * kKVBytes;
constexpr int kStashOff = kPOff + kBufs * kPBytes;     // [kStash][128] o, then [kStash] m, l
constexpr int kCtlOff = kStashOff + kStash * (kDH + 2) * 4;
constexpr int kRunSlots = 4;
constexpr int kQLoadBytes = 2 * 2 * 64 * 2;            // query rows 0-1 of both 64-dim boxes
constexpr int kTmemCols = 128;                         // kBufs buffers of (S: 16, O: 16)
constexpr int kThreads = 384;
constexpr int kSoftmaxWarp0 = 4;
constexpr int kEpilogueWarp0 = 8;

// Unit v (the v-th unit of this CTA with keys) uses K stage v % kKStages, V stage
// v % kVStages and TMEM/P buffer v % kBufs; every barrier completes once per use of its
// stage or buffer, with parity (v / depth) & 1.
struct Ctl {
  uint64_t kfull[kKStages], kempty[kKStages];   // K + query stage landed / free (after S)
  uint64_t vfull[kVStages], vempty[kVStages];   // V stage landed / free (after O)
  uint64_t sfull[kBufs], sfree[kBufs], pfull[kBufs], ofull[kBufs], ofree[kBufs];
  uint64_t rfull[kRunSlots], rempty[kRunSlots];
  float red_m[4], red_l[4];
  float ml[kBufs][2];
  int run[kRunSlots][3];
  uint32_t tmem;
  int abort;
};
constexpr int kSmem = kCtlOff + (int)sizeof(Ctl) + 1024;   // + base alignment
static_assert(kSmem <= 227 * 1024, "tensor-core attention shared memory");
static_assert(kAttnChunk == 128, "one MMA tile of keys per unit");

// byte offset of element (row, col) of a [rows][64] bf16 tile in the 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int row, int col) {
  const uint32_t b = (uint32_t)col * 2;
  return (uint32_t)row * 128 + ((((b >> 4) ^ (uint32_t)(row & 7)) << 4) | (b & 15));
}

__device__ __forceinline__ bool wait_or_flag(uint32_t bar, uint32_t parity, const AttnArgs& a,
                                             volatile int* abort_flag) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity, a.test_ctl)) return true;
  raise_timeout(a, abort_flag);
  return false;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_attn_tc(const AttnArgs a, int units, int slot_base, const __grid_constant__ CUtensorMap mapK,
              const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapQ) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kCtlOff);
  volatile int* abort_flag = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u0 = (int)(((long long)blockIdx.x * units) / gridDim.x);
  const int u1 = (int)(((long long)(blockIdx.x + 1) * units) / gridDim.x);
  auto B32 = [](uint64_t& b) { return smem_u32(&b); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(B32(ctl->kfull[i]), 1);
      mbar_init(B32(ctl->kempty[i]), 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(B32(ctl->vfull[i]), 1);
      mbar_init(B32(ctl->vempty[i]), 1);
    }
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(B32(ctl->sfull[i]), 1);
      mbar_init(B32(ctl->sfree[i]), 4);   // one arrival per warp of the warpgroup
      mbar_init(B32(ctl->pfull[i]), 4);
      mbar_init(B32(ctl->ofull[i]), 1);
      mbar_init(B32(ctl->ofree[i]), 4);
    }
    for (int i = 0; i < kRunSlots; ++i) {
      mbar_init(B32(ctl->rfull[i]), 4);
      mbar_init(B32(ctl->rempty[i]), 1);
    }
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = ctl->tmem;
  pdl_wait_and_trigger();
  if (a.early_trigger) pdl_trigger();

  auto next_valid = [&](int u) {
    while (u < u1 && decode_unit(a, u).nk == 0) ++u;
    return u;
  };

  if (warp == 0) {
    // ---- TMA producer: K + query and V of each unit, as far ahead as their rings allow;
    // V never ahead of K.  Non-blocking polls; bounded idle time.
    if (lane == 0) {
      int vk = 0, vv = 0;
      int uk = next_valid(u0), uv = uk;
      uint32_t idle = 0, idle_limit = 4 * kWaitLimit;
      int32_t armed, kinds;
      read_withhold(a.test_ctl, armed, kinds);
      while ((uk < u1 || uv < u1) && !*abort_flag) {
        bool progressed = false;
        if (uk < u1 && (vk < kKStages || mbar_test(B32(ctl->kempty[vk % kKStages]),
                                                   ((vk / kKStages) - 1) & 1))) {
          const Unit t = decode_unit(a, uk);
          const uint32_t sb = smem_u32(smem + (vk % kKStages) * kKStageBytes);
          const uint32_t full = B32(ctl->kfull[vk % kKStages]);
          const int row = t.c * kAttnChunk, sc = slot_base + t.s;
          const int qrow = (t.s * a.H + t.h) * 2;
          mbar_expect_tx(full, kKVBytes + kQLoadBytes);
          tma_load_4d(sb, &mapK, 0, row, t.h, sc, full);
          tma_load_4d(sb + kBoxBytes, &mapK, 64, row, t.h, sc, full);
          tma_load_2d(sb + kKVBytes, &mapQ, 0, qrow, full);
          tma_load_2d(sb + kKVBytes + kQBoxBytes, &mapQ, 64, qrow, full);
          ++vk;
          uk = next_valid(uk + 1);
          progressed = true;
        }
        if (uv < u1 && vv < vk && (vv < kVStages || mbar_test(B32(ctl->vempty[vv % kVStages]),
                                                              ((vv / kVStages) - 1) & 1))) {
          const Unit t = decode_unit(a, uv);
          const uint32_t vb = smem_u32(smem + kVOff + (vv % kVStages) * kKVBytes);
          const uint32_t full = B32(ctl->vfull[vv % kVStages]);
          const int row = t.c * kAttnChunk, sc = slot_base + t.s;
          // a failure-detection test may have this producer withhold its first V tile:
          // that stage never completes and the MMA issuer's bounded polling runs out
          if (!(vv == 0 && take_withhold(a.test_ctl, armed, kinds, PP_TEST_ATTN))) {
            mbar_expect_tx(full, kKVBytes);
            tma_load_4d(vb, &mapV, 0, row, t.h, sc, full);
            tma_load_4d(vb + kBoxBytes, &mapV, 64, row, t.h, sc, full);
          }
          ++vv;
          uv = next_valid(uv + 1);
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else if (++idle > idle_limit) {
          raise_timeout(a, abort_flag);
        } else if (idle == kWaitFastPolls) {
          idle_limit = 4 * wait_budget(a.test_ctl);
        }
      }
      // every copy this CTA issued lands before the CTA may exit (bounded waits)
      for (int i = vk > kKStages ? vk - kKStages : 0; i < vk; ++i)
        mbar_wait(B32(ctl->kfull[i % kKStages]), (i / kKStages) & 1, a.test_ctl);
      for (int i = vv > kVStages ? vv - kVStages : 0; i < vv; ++i)
        mbar_wait(B32(ctl->vfull[i % kVStages]), (i / kVStages) & 1, a.test_ctl);
    }
  } else if (warp == 1) {
    // ---- MMA issuer ---------------------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t id_s = instr_desc(128, 16);               // K-major A and B
      constexpr uint32_t id_o = instr_desc(128, 16) | (1u << 15);  // A (V^T) MN-major
      // Issue whichever is ready: the scores of unit vq (at most kBufs - 1 units ahead
      // of the outputs) or the output of unit vp.  Polls are non-blocking so that
      // neither waits behind the other; a bounded number of idle polls raises the timeout.
      int vq = 0, vp = 0;
      int uq = next_valid(u0);
      uint32_t idle = 0, idle_limit = 4 * kWaitLimit;
      // barrier and parity of the most recent commit: MMAs complete in issue order, so
      // once it has arrived every MMA of this CTA is done
      uint32_t last_bar = 0, last_par = 0;
      while ((uq < u1 || vp < vq) && !*abort_flag) {
        bool progressed = false;
        if (uq < u1 && vq < vp + kBufs) {
          const int i = vq % kBufs, ks = vq % kKStages;
          if (mbar_test(B32(ctl->kfull[ks]), (vq / kKStages) & 1) &&
              (vq < kBufs || mbar_test(B32(ctl->sfree[i]), ((vq / kBufs) - 1) & 1))) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t kb = smem_u32(smem + ks * kKStageBytes);
            const uint32_t qb = kb + kKVBytes;
#pragma unroll
            for (int kk = 0; kk < kDH / 16; ++kk) {
              const uint32_t ko = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
              const uint32_t qo = (kk >> 2) * kQBoxBytes + (kk & 3) * 32;
              umma_bf16(tmem + 32 * i, smem_desc(kb + ko), smem_desc(qb + qo), id_s,
                        kk > 0 ? 1u : 0u);
            }
            umma_commit(B32(ctl->sfull[i]));
            umma_commit(B32(ctl->kempty[ks]));
            last_bar = B32(ctl->sfull[i]);
            last_par = (vq / kBufs) & 1;
            ++vq;
            uq = next_valid(uq + 1);
            progressed = true;
          }
        }
        if (vp < vq) {
          const int i = vp % kBufs, vs = vp % kVStages;
          if (mbar_test(B32(ctl->pfull[i]), (vp / kBufs) & 1) &&
              mbar_test(B32(ctl->vfull[vs]), (vp / kVStages) & 1) &&
              (vp < kBufs || mbar_test(B32(ctl->ofree[i]), ((vp / kBufs) - 1) & 1))) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t vb = smem_u32(smem + kVOff + vs * kKVBytes);
            const uint32_t pb = smem_u32(smem + kPOff + i * kPBytes);
#pragma unroll
            for (int kk = 0; kk < kAttnChunk / 16; ++kk) {
              const uint32_t po = (kk >> 2) * kQBoxBytes + (kk & 3) * 32;
              // 16 keys = two 8-key atoms (1024 bytes apart); dims 64..127 one box further
              umma_bf16(tmem + 32 * i + 16, smem_desc_mn(vb + kk * 2048, kBoxBytes),
                        smem_desc(pb + po), id_o, kk > 0 ? 1u : 0u);
            }
            umma_commit(B32(ctl->ofull[i]));
            umma_commit(B32(ctl->vempty[vs]));
            last_bar = B32(ctl->ofull[i]);
            last_par = (vp / kBufs) & 1;
            ++vp;
            progressed = true;
          }
        }
        if (progressed) {
          idle = 0;
        } else if (++idle > idle_limit) {
          raise_timeout(a, abort_flag);
        } else if (idle == kWaitFastPolls) {
          idle_limit = 4 * wait_budget(a.test_ctl);
        }
      }
      // the last MMAs complete before the tensor memory is released (also after a
      // timeout, when score MMAs may have been issued after the last output MMA)
      if (vq > 0) mbar_wait(last_bar, last_par, a.test_ctl);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ---- merge warp: tickets and final merges ------------------------------------------
    // lane 0 waits and reads the run; the warp follows it (uniform control flow)
    for (int r = 0;; ++r) {
      const int q = r % kRunSlots;
      int pair = -1, len = 0, nc = 0;
      if (lane == 0 && wait_or_flag(B32(ctl->rfull[q]), (r / kRunSlots) & 1, a, abort_flag)) {
        pair = ctl->run[q][0];
        len = ctl->run[q][1];
        nc = ctl->run[q][2];
        if (pair >= (units / a.nc_max)) pair = -1;   // never index past the pairs
      }
      pair = __shfl_sync(0xffffffffu, pair, 0);
      len = __shfl_sync(0xffffffffu, len, 0);
      nc = __shfl_sync(0xffffffffu, nc, 0);
      if (pair < 0) break;   // end of this CTA's runs (or a wait gave up)
      unsigned last = 0;
      if (lane == 0) {
        __threadfence();   // the epilogue's partial stores (ordered by the barrier) first
        const unsigned prev = atomicAdd(a.count + pair, (unsigned)len);
        last = (prev + (unsigned)len == (unsigned)nc);
        mbar_arrive(B32(ctl->rempty[q]));
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence();
        const int s = pair / a.H, h = pair - s * a.H;
        merge_pair<kDH>(a, a.part + (size_t)pair * attn_pair_floats(a.nc_max, kDH), nc, s, h,
                        lane);
        if (lane == 0) a.count[pair] = 0u;
      }
    }
  } else if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 4) {
    // ---- softmax: thread t = key t of the chunk --------------------------------------
    const int wq = warp - kSoftmaxWarp0;
    const int key = threadIdx.x - kSoftmaxWarp0 * 32;
    int v = 0;
    for (int u = u0; u < u1; ++u) {
      const Unit t = decode_unit(a, u);
      if (t.nk == 0) continue;
      const int bb = v % kBufs;
      const uint32_t ph = (v / kBufs) & 1;
      wait_or_flag(B32(ctl->sfull[bb]), ph, a, abort_flag);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      uint32_t r[2];
      tmem_ld2(tmem + ((uint32_t)(wq * 32) << 16) + 32 * bb, r);
      tmem_wait_ld();
      const float sv = after_wait(r[0]) + after_wait(r[1]);
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(B32(ctl->sfree[bb]));
      const bool valid = key < t.nk;
      float m = valid ? sv : -INFINITY;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) ctl->red_m[wq] = m;
      named_sync(1, 128);
      const float M = fmaxf(fmaxf(ctl->red_m[0], ctl->red_m[1]), fmaxf(ctl->red_m[2], ctl->red_m[3]));
      const float p = valid ? exp2f(sv - M) : 0.f;
      float l = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (lane == 0) ctl->red_l[wq] = l;
      named_sync(1, 128);
      const float L = ((ctl->red_l[0] + ctl->red_l[1]) + ctl->red_l[2]) + ctl->red_l[3];
      // P and (max, sum) of this buffer are free once the epilogue of its last unit is done
      if (v >= kBufs) wait_or_flag(B32(ctl->ofree[bb]), ph ^ 1, a, abort_flag);
      uint16_t p_hi, p_lo;
      bf16_split(p, p_hi, p_lo);
      uint8_t* pt = smem + kPOff + bb * kPBytes + (key >> 6) * kQBoxBytes;
      *reinterpret_cast<uint16_t*>(pt + sw128(0, key & 63)) = p_hi;
      *reinterpret_cast<uint16_t*>(pt + sw128(1, key & 63)) = p_lo;
      if (t.nk < kAttnChunk) {
        // ragged chunk: V rows past the valid keys may hold anything (even NaN); zero
        // them so that p = 0 contributes exactly nothing
        wait_or_flag(B32(ctl->vfull[v % kVStages]), (v / kVStages) & 1, a, abort_flag);
        if (!valid) {
          uint8_t* vr = smem + kVOff + (v % kVStages) * kKVBytes + key * 128;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            *reinterpret_cast<uint4*>(vr + i * 16) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vr + kBoxBytes + i * 16) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      if (key == 0) {
        ctl->ml[bb][0] = M;
        ctl->ml[bb][1] = L;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(B32(ctl->pfull[bb]));
      ++v;
    }
  } else if (warp >= kEpilogueWarp0) {
    // ---- epilogue: thread t = output dim t -------------------------------------------
    // A (slot, head) whose chunks all fall in this CTA's unit range is merged here from
    // the on-chip stash; the others go through global partials and the merge warp.  Both
    // merges do the same arithmetic in the same order, so the bits do not depend on
    // which one ran.
    const int wq = warp - kEpilogueWarp0;
    const int dim = threadIdx.x - kEpilogueWarp0 * 32;
    const int HD = a.H * kDH;
    float* st_o = reinterpret_cast<float*>(smem + kStashOff);   // [kStash][kDH]
    float* st_m = st_o + kStash * kDH;                           // [kStash]
    float* st_l = st_m + kStash;                                 // [kStash]
    const bool stash_ok = a.nc_max <= kStash;
    int v = 0, runs = 0, run_pair = -1, run_len = 0, run_nc = 0;
    bool run_local = false;
    auto enqueue = [&](int pair, int len, int nc) {
      const int q = runs % kRunSlots;
      if (runs >= kRunSlots)
        wait_or_flag(B32(ctl->rempty[q]), ((runs / kRunSlots) - 1) & 1, a, abort_flag);
      if (dim == 0) {
        ctl->run[q][0] = pair;
        ctl->run[q][1] = len;
        ctl->run[q][2] = nc;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(B32(ctl->rfull[q]));
      ++runs;
    };
    auto finish_run = [&]() {
      if (run_len == 0) return;
      if (run_local) {
        named_sync(2, 128);   // the stash holds every chunk of the pair
        float M = -INFINITY;
        for (int c = 0; c < run_nc; ++c) M = fmaxf(M, st_m[c]);
        float L = 0.f, O = 0.f;
        for (int c = 0; c < run_nc; ++c) {
          const float f = exp2f(st_m[c] - M);
          L = fmaf(f, st_l[c], L);
          O = fmaf(f, st_o[c * kDH + dim], O);
        }
        const int s = run_pair / a.H, h = run_pair - s * a.H;
        const float r = O / L;
        a.out[(size_t)s * a.out_ld + h * kDH + dim] = r;
        if (a.op) op_store(a.op, HD, a.op_Bp, s, h * kDH + dim, r);
        named_sync(2, 128);   // the stash is free for the next pair
      } else {
        enqueue(run_pair, run_len, run_nc);
      }
      run_len = 0;
    };
    for (int u = u0; u < u1; ++u) {
      const Unit t = decode_unit(a, u);
      const int pair = t.s * a.H + t.h;
      if (t.nk == 0) {
        if (t.c == 0) {   // closed slot: zero output
          a.out[(size_t)t.s * a.out_ld + t.h * kDH + dim] = 0.f;
          if (a.op) op_store(a.op, HD, a.op_Bp, t.s, t.h * kDH + dim, 0.f);
        }
        continue;
      }
      if (pair != run_pair) {
        finish_run();
        run_pair = pair;
        run_nc = (min(__ldg(a.n_valid + t.s), a.W) + kAttnChunk - 1) / kAttnChunk;
        const int first = pair * a.nc_max;   // the pair's valid units: first .. first+nc-1
        run_local = stash_ok && first >= u0 && first + run_nc <= u1;
      }
      const int bb = v % kBufs;
      const uint32_t ph = (v / kBufs) & 1;
      wait_or_flag(B32(ctl->ofull[bb]), ph, a, abort_flag);
      wait_or_flag(B32(ctl->pfull[bb]), ph, a, abort_flag);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      uint32_t r[2];
      tmem_ld2(tmem + ((uint32_t)(wq * 32) << 16) + 32 * bb + 16, r);
      tmem_wait_ld();
      const float o = after_wait(r[0]) + after_wait(r[1]);
      const float mc = ctl->ml[bb][0], lc = ctl->ml[bb][1];
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(B32(ctl->ofree[bb]));
      if (run_local) {
        st_o[t.c * kDH + dim] = o;
        if (dim == 0) {
          st_m[t.c] = mc;
          st_l[t.c] = lc;
        }
      } else {
        float* dst = a.part + (size_t)pair * attn_pair_floats(a.nc_max, kDH) +
                     (size_t)t.c * attn_rec_floats(kDH);
        dst[8 + dim] = o;
        if (dim < 8) dst[dim] = dim == 0 ? mc : (dim == 1 ? lc : 0.f);   // whole sector
      }
      ++run_len;
      ++v;
    }
    finish_run();
    enqueue(-1, 0, 0);
  }

  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  pdl_trigger();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols));
  }
}

__global__ void k_q_split(const float* q, int q_ld, float scale, int H, uint16_t* q_op) {
  pdl_wait_and_trigger();
  const int pair = blockIdx.x, s = pair / H, h = pair - s * H, i = threadIdx.x;
  const float v = q[(size_t)s * q_ld + h * kDH + i] * scale;
  uint16_t hi, lo;
  bf16_split(v, hi, lo);
  q_op[((size_t)pair * 2) * kDH + i] = hi;
  q_op[((size_t)pair * 2 + 1) * kDH + i] = lo;
}

}  // namespace

cudaError_t launch_attn_tc(const AttnArgs& a, int B, const AttnMaps& maps, int slot_base,
                           cudaStream_t s) {
  if (B < 1 || a.H < 1 || a.nc_max < 1) return cudaErrorInvalidValue;
  cudaError_t err =
      cudaFuncSetAttribute(k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (err != cudaSuccess) return err;
  const int units = B * a.H * a.nc_max;
  const int nsm = attn::sm_count();
  const int grid = units < nsm ? units : nsm;
  return launch_k(k_attn_tc, dim3(grid), dim3(kThreads), (size_t)kSmem, s, 1, a, units, slot_base,
                  maps.k, maps.v, maps.q);
}

cudaError_t launch_q_split(const AttnArgs& a, int B, int Dh, cudaStream_t s) {
  if (Dh != kDH || !a.q_op) return cudaErrorInvalidValue;
  return launch_k(k_q_split, dim3(B * a.H), dim3(kDH), 0, s, 1, a.q, a.q_ld, a.q_scale, a.H,
                  a.q_op);
}

}  // namespace pp
