// pp_api.cu - the C ABI (include/pp.h): engine creation over caller-owned weights and
// workspace, the session table, and one lockstep tick captured as a CUDA graph.
#include <math.h>
#include <string.h>

#include <cmath>

#include <new>
#include <vector>

#include "pp_internal.cuh"
#include "pp_sample.cuh"

using namespace pp;

namespace pp {
bool g_use_pdl = false;
int g_launch_priority = 0;
}

// Timing events recorded at every kernel boundary of the profiling graph.
struct Prof {
  std::vector<cudaEvent_t> ev;
  std::vector<int> kind;           // kind of the kernel that starts at ev[i]
  cudaError_t mark(int k, cudaStream_t s) {
    cudaEvent_t e;
    cudaError_t err = cudaEventCreate(&e);
    if (err != cudaSuccess) return err;
    ev.push_back(e);
    kind.push_back(k);
    return cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  }
  void clear() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    ev.clear();
    kind.clear();
  }
};

// One family of tensor-core contractions (one stacked weight tensor).
struct Mm {
  CUtensorMap mapA;    // stacked weights [rows_total, K] bf16, box 64 k x 128 rows
                       // (gate/up pairs: 64 rows)
  CUtensorMap mapB;    // activation operand [2*Bp, K] bf16, box 64 k x 2*Bp rows
  int M = 0, K = 0, kblocks = 0, splits = 1, m_tiles = 0, pair = 0;
  int H = 1;           // 128-row halves per weight tile
};

enum MmKind { MM_QKV, MM_O, MM_GU, MM_DOWN, MM_TEXT, MM_DIN, MM_DQKV, MM_DO, MM_DGU, MM_DDOWN,
              MM_DHEAD,
              // the depformer's batched user steps: one chunk of operand rows per step
              MM_BDQKV, MM_BDO, MM_BDGU, MM_BDDOWN, MM_BDHEAD, MM_COUNT };

constexpr int kMaxGroups = 2;

// A group is a contiguous range of slots run as one independent chain of kernels (its
// own ring, activations, operands and contraction plans).  With two groups the tick
// graph has two parallel branches: one group's latency-bound depformer overlaps the
// other group's bandwidth-bound attention.  Every kernel computes each slot the same
// way whatever the group size, so grouping does not change any session's bits.
struct Group {
  int slot0 = 0;
  bool wide_tiles = false;  // 256-row weight tiles for the large temporal matrices
  Dims D;
  Buffers buf;
  Mm mm[MM_COUNT];
  AttnMaps amaps;        // ring and query operand maps of the tensor-core attention
  bool has_amaps = false;
};

struct pp_engine {
  pp_config cfg;
  int B = 0;             // all slots
  int ngroups = 1;
  Group grp[kMaxGroups];
  Buffers shared;        // per-slot state and staging for all slots (group 0 base)
  int logits_ld = 0;
  int dep_priority = 0;  // launch priority of the depformer kernels (higher = more urgent)
  bool tensor = true;
  bool pdl = true;
  cudaStream_t branch[kMaxGroups] = {nullptr, nullptr};
  cudaEvent_t fork = nullptr, join[kMaxGroups] = {nullptr, nullptr};
  cudaStream_t cap_stream = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;      // the tick with the decision kernels (sampling)
  cudaGraph_t graph_greedy = nullptr;
  cudaGraphExec_t exec_greedy = nullptr;   // greedy decisions fused into the heads
  int n_kernels = 0;
  cudaGraph_t prof_graph = nullptr;
  cudaGraphExec_t prof_exec = nullptr;
  Prof prof;
  std::vector<int32_t> ctl, ctl_pos;   // uploaded before the next tick when dirty
  bool ctl_dirty = false;
  std::vector<SampleParams> samp;      // per-slot sampling parameters, uploaded when dirty
  bool samp_dirty = false;
  std::vector<int64_t> pos;            // host mirror of each open slot's position
  std::vector<uint8_t> open;
  int32_t test_word[4] = {0, 0, 0, 0};  // host copy of the fault-test word
};

namespace {

bool head_dim_ok(int hd) { return hd == 32 || hd == 64 || hd == 128; }

bool config_ok(const pp_config* c) {
  if (!c) return false;
  if (c->d_model <= 0 || c->n_layers <= 0 || c->n_heads <= 0 || c->ffn <= 0) return false;
  if (c->d_model % c->n_heads || !head_dim_ok(c->d_model / c->n_heads)) return false;
  if (c->dep_d <= 0 || c->dep_layers <= 0 || c->dep_heads <= 0 || c->dep_ffn <= 0) return false;
  if (c->dep_d % c->dep_heads || !head_dim_ok(c->dep_d / c->dep_heads)) return false;
  // one warp per depformer head in one CTA, within the step attention's register budget
  if (c->dep_heads > kDepAttnMaxHeads(c->dep_d / c->dep_heads)) return false;
  if (c->n_q != 16 || c->text_vocab <= 0 || c->audio_card <= 0) return false;
  if (c->window <= 0 || c->max_batch <= 0 || c->max_batch > kMaxBatch) return false;
  // 16-byte rows for the vectorised weight and activation streams
  if (c->d_model % 8 || c->ffn % 8 || c->dep_d % 8 || c->dep_ffn % 8) return false;
  if (!(c->eps > 0.f) || !(c->rope_base > 1.f)) return false;
  // the persistent depformer serves small engines on the tensor-core path
  if ((c->flags & PP_FLAG_LOW_LATENCY) &&
      (c->max_batch > kPMaxB || (c->flags & PP_FLAG_CUDA_CORE_GEMM)))
    return false;
  return true;
}

Dims make_dims(const pp_config* c) {
  Dims D;
  D.Bp = (c->max_batch + 7) / 8 * 8;
  D.d = c->d_model; D.L = c->n_layers; D.H = c->n_heads; D.Dh = c->d_model / c->n_heads;
  D.F = c->ffn; D.Vt = c->text_vocab; D.Va = c->audio_card; D.nq = c->n_q;
  D.dd = c->dep_d; D.Ld = c->dep_layers; D.Hd = c->dep_heads; D.Dhd = c->dep_d / c->dep_heads;
  D.Fd = c->dep_ffn; D.W = c->window; D.B = c->max_batch;
  D.eps = c->eps; D.rope_base = c->rope_base;
  D.nc_max = (c->window + kAttnChunk - 1) / kAttnChunk;
  D.logits_ld = c->text_vocab + c->n_q * c->audio_card;
  // the user steps run as one batched pass on the tensor-core path unless elided or
  // asked to run one at a time
  const bool tensor = !(c->flags & PP_FLAG_CUDA_CORE_GEMM);
  D.dep_persist = tensor && (c->flags & PP_FLAG_LOW_LATENCY);
  D.dep_batched = tensor && !D.dep_persist &&
                  !(c->flags & (PP_FLAG_SKIP_USER_STEPS | PP_FLAG_SEQUENTIAL_USER_STEPS));
  D.dep_steps = ((c->flags & PP_FLAG_SKIP_USER_STEPS) || D.dep_batched) ? c->n_q / 2 : c->n_q;
  if (D.dep_persist) D.dep_steps = 0;   // every step runs inside the persistent kernel
  D.samp_text = (int64_t)c->text_vocab * 4 <= kSampleSmemMax;
  D.samp_audio = (int64_t)c->audio_card * 4 <= kSampleSmemMax;
  return D;
}

// Workspace carve-up: every region 256-byte aligned, in a fixed order.
struct Carver {
  char* base;
  size_t off = 0;
  template <class T>
  T* take(size_t count) {
    off = (off + 255) & ~(size_t)255;
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

int group_count(const pp_config* c) {
  return (c->max_batch >= 16 && (c->flags & PP_FLAG_TWO_GROUPS)) ? 2 : 1;
}

// Workspace layout: per-slot state and staging for all slots first, then each group's
// ring, activations and operands.  Fills shared and grp[] (pointers) when base != 0.
size_t carve(const pp_config* c, char* base, Buffers* shared, Group* grp) {
  Carver cv{base};
  const size_t B = c->max_batch;
  const int ng = group_count(c);
  const size_t ld = (size_t)c->text_vocab + (size_t)c->n_q * c->audio_card;
  Buffers sh{};
  sh.pos = cv.take<int32_t>(B);
  sh.live = cv.take<int32_t>(B);
  sh.nvalid = cv.take<int32_t>(B);
  sh.ctl = cv.take<int32_t>(B);
  sh.ctl_pos = cv.take<int32_t>(B);
  sh.status = cv.take<uint32_t>(1);
  sh.test_ctl = cv.take<int32_t>(4);
  sh.samp = cv.take<SampleParams>(B);
  sh.hist_len = cv.take<int32_t>(B);
  sh.hist = cv.take<int32_t>(B * kHist);
  sh.in_col = cv.take<int32_t>(B * kRows);
  sh.in_user = cv.take<int32_t>(B * PP_USER_ROWS);
  sh.in_fmask = cv.take<uint8_t>(B * kRows);
  sh.in_forced = cv.take<int32_t>(B * kRows);
  sh.out_col = cv.take<int32_t>(B * kRows);
  sh.logits = cv.take<float>(B * ld);
  if (shared) *shared = sh;
  int slot0 = 0;
  for (int g = 0; g < ng; ++g) {
    const int Bg = (g == 0) ? (int)(B + ng - 1) / ng : (int)B - slot0;
    pp_config cg = *c;
    cg.max_batch = Bg;
    const Dims D = make_dims(&cg);
    Buffers b = sh;   // per-slot state: this group's slice
    if (base) {
      b.pos = sh.pos + slot0;
      b.live = sh.live + slot0;
      b.nvalid = sh.nvalid + slot0;
      b.ctl = sh.ctl + slot0;
      b.ctl_pos = sh.ctl_pos + slot0;
      b.samp = sh.samp + slot0;
      b.hist_len = sh.hist_len + slot0;
      b.hist = sh.hist + (size_t)slot0 * kHist;
      b.in_col = sh.in_col + (size_t)slot0 * kRows;
      b.in_user = sh.in_user + (size_t)slot0 * PP_USER_ROWS;
      b.in_fmask = sh.in_fmask + (size_t)slot0 * kRows;
      b.in_forced = sh.in_forced + (size_t)slot0 * kRows;
      b.out_col = sh.out_col + (size_t)slot0 * kRows;
      b.logits = sh.logits + (size_t)slot0 * ld;
    }
    const size_t Bs = Bg;
    const size_t wide = D.d > D.F ? D.d : D.F;
    const size_t dwide = D.dd > D.Fd ? D.dd : D.Fd;
    b.ring = cv.take<uint16_t>((size_t)D.L * Bs * 2 * D.H * D.W * D.Dh);
    b.attn_count = cv.take<uint32_t>(Bs * D.H);
    b.x = cv.take<float>(Bs * D.d);
    b.xn = cv.take<float>(Bs * wide);
    b.z = cv.take<float>(Bs * D.d);
    b.qkv = cv.take<float>(Bs * 3 * D.d);
    b.q = cv.take<float>(Bs * D.d);
    b.q_op = cv.take<uint16_t>(Bs * D.H * 2 * D.Dh);
    b.o = cv.take<float>(Bs * D.d);
    b.hmlp = cv.take<float>(Bs * D.F);
    b.rope_cs = cv.take<float>(Bs * D.Dh);
    b.attn_part = cv.take<float>(Bs * D.H * attn_pair_floats(D.nc_max, D.Dh));
    b.tok = cv.take<int32_t>(Bs);
    b.y = cv.take<float>(Bs * D.dd);
    b.yn = cv.take<float>(Bs * dwide);
    b.dqkv = cv.take<float>(Bs * 3 * D.dd);
    b.dkv = cv.take<float>(Bs * D.Ld * D.nq * 2 * D.dd);
    b.dout = cv.take<float>(Bs * D.dd);
    b.dh = cv.take<float>(Bs * D.Fd);
    b.tokb = cv.take<int32_t>(kDepBatch * Bs);
    b.y_b = cv.take<float>(kDepBatch * Bs * D.dd);
    b.pz = cv.take<float>(Bs * D.nq * D.dd);
    b.dqkv_b = cv.take<float>(kDepBatch * Bs * 3 * D.dd);
    b.dout_b = cv.take<float>(kDepBatch * Bs * D.dd);
    const size_t R = 2 * (size_t)D.Bp;
    b.op_d = cv.take<uint16_t>(R * D.d);
    b.op_o = cv.take<uint16_t>(R * D.d);
    b.op_f = cv.take<uint16_t>(R * D.F);
    b.op_z = cv.take<uint16_t>(R * D.d);
    b.op_dd = cv.take<uint16_t>(R * D.dd);
    b.op_do = cv.take<uint16_t>(R * D.dd);
    b.op_fd = cv.take<uint16_t>(R * D.Fd);
    b.op_ddb = cv.take<uint16_t>(kDepBatch * R * D.dd);
    b.op_dob = cv.take<uint16_t>(kDepBatch * R * D.dd);
    b.op_fdb = cv.take<uint16_t>(kDepBatch * R * D.Fd);
    b.ssq = cv.take<float>((size_t)kMaxUnits * Bs);
    b.rstd_z = cv.take<float>(Bs);
    b.dkey = cv.take<unsigned long long>(2 * Bs);
    b.dnan = cv.take<unsigned>(2);
    b.dticket = cv.take<unsigned>(4);
    b.pbar = cv.take<unsigned>(4);
    b.ppart_val = cv.take<float>((size_t)kPMaxGrid * kPMaxB);
    b.ppart_idx = cv.take<int>((size_t)kPMaxGrid * kPMaxB);
    if (grp) {
      grp[g].slot0 = slot0;
      grp[g].D = D;
      grp[g].buf = b;
    }
    slot0 += Bg;
  }
  return (cv.off + 255) & ~(size_t)255;
}

#define PP_TRY(x)                         \
  do {                                    \
    cudaError_t err_ = (x);               \
    if (err_ != cudaSuccess) return err_; \
  } while (0)


// ---- tensor maps and contraction plans ------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D bf16 map over a row-major [rows, k] matrix, 64-element (128-byte) inner box with
// the 128-byte swizzle; out-of-range rows and columns read as zero.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t k, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[2] = {k, rows};
  cuuint64_t gstride[1] = {k * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// K and V as 4-D [slots][H][W][Dh] (slot stride in elements), box 64 dims x 128 ring rows;
// the query operand as 2-D [pairs*2][Dh], box 64 x 2 rows.  Rows past W (or past the
// last query row) read as zero.
bool pp::attn_maps(AttnMaps* m, const uint16_t* k, const uint16_t* v, size_t slot_stride, int slots,
               int H, int W, int Dh, const uint16_t* q_op, int pairs) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || Dh != 128) return false;
  cuuint64_t gdim[4] = {(cuuint64_t)Dh, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)slots};
  cuuint64_t gstride[3] = {(cuuint64_t)Dh * 2, (cuuint64_t)W * Dh * 2, (cuuint64_t)slot_stride * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)kAttnChunk, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  for (int i = 0; i < 2; ++i) {
    if (fn(i == 0 ? &m->k : &m->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
           const_cast<uint16_t*>(i == 0 ? k : v), gdim, gstride, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  cuuint64_t qdim[2] = {(cuuint64_t)Dh, (cuuint64_t)pairs * 2};
  cuuint64_t qstride[1] = {(cuuint64_t)Dh * 2};
  cuuint32_t qbox[2] = {64, 2};   // rows hi, lo of one (slot, head); the other operand rows
                                  // of the MMA tile feed output columns that are never read
  return fn(&m->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(q_op), qdim, qstride,
            qbox, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// K-splits per M-tile: a function of the matrix shape and the device's SM count only,
// never of the batch, so every engine size reduces in the same order.  Model: units run
// in waves of two CTAs per SM; a unit costs its k-blocks plus a fixed overhead of about
// five k-blocks (launch share, pipeline fill, epilogue; calibrated on GB300 by sweeping
// the split counts of the full-size matrices at 64 slots) plus half a k-block per split
// (the cluster reduction grows with the splits; this moved the small depformer
// contractions from 8 to 4 splits, -0.25 ms per B=64 tick on GB300).
int choose_splits(int m_tiles, int kblocks, int nsm, int per_sm) {
  const int slots = per_sm * nsm;
  int best = 1;
  double best_t = 1e300;
  for (int sp = 1; sp <= kblocks && sp <= kMaxSplits && m_tiles * sp <= kMaxUnits; ++sp) {
    const int units = m_tiles * sp;
    const int waves = (units + slots - 1) / slots;
    const double t = waves * ((double)((kblocks + sp - 1) / sp) + 5.0 + 0.5 * sp);
    if (t < best_t - 1e-9) { best_t = t; best = sp; }
  }
  return best;
}

// chunks: column chunks of one launch (the split count accounts for all of them);
// op_chunks: operand chunks the B map spans (1 when the chunks share one operand);
// H: 128-row halves per weight tile (a function of the matrix shape only, so that every
// engine size reduces in the same order)
bool plan_mm(Mm* g, const void* w, int rows_total, int M, int K, int pair, const uint16_t* op,
             int Bp, int nsm, int chunks = 1, int op_chunks = 1, int H = 1) {
  g->M = M;
  g->K = K;
  g->pair = pair;
  g->H = H;
  // the split-K epilogue moves rows in aligned groups of 4
  if (!pair && M % 4) return false;
  g->kblocks = (K + 63) / 64;
  g->m_tiles = pair ? (pair + 64 * H - 1) / (64 * H) : (M + 128 * H - 1) / (128 * H);
  if (g->m_tiles > kMaxTiles) return false;
  g->splits = choose_splits(g->m_tiles * chunks, g->kblocks, nsm, H == 1 ? 2 : 1);
  // weight boxes: 128 rows (one 16 KB copy each), or 64 rows for the gate/up pairs of a
  // 128-row tile
  return make_map(&g->mapA, w, (uint64_t)rows_total, (uint64_t)K, (pair && H == 1) ? 64 : 128) &&
         make_map(&g->mapB, op, (uint64_t)op_chunks * 2 * Bp, (uint64_t)K, 2 * Bp);
}

bool plan_all(Group* e, int nsm) {
  const Dims& D = e->D;
  const Buffers& b = e->buf;
  const int Bp = D.Bp;
  bool ok = true;
  // with wide tiles, the temporal layers' matrices and the text head take 256-row tiles
  // whose halves share each activation tile
  const int Ht = e->wide_tiles ? 2 : 1;
  ok &= plan_mm(&e->mm[MM_QKV], b.wqkv, D.L * 3 * D.d, 3 * D.d, D.d, 0, b.op_d, Bp, nsm, 1, 1, Ht);
  ok &= plan_mm(&e->mm[MM_O], b.wo, D.L * D.d, D.d, D.d, 0, b.op_o, Bp, nsm, 1, 1, Ht);
  ok &= plan_mm(&e->mm[MM_GU], b.wgu, D.L * 2 * D.F, D.F, D.d, D.F, b.op_d, Bp, nsm, 1, 1, Ht);
  ok &= plan_mm(&e->mm[MM_DOWN], b.wdown, D.L * D.d, D.d, D.F, 0, b.op_f, Bp, nsm, 1, 1, Ht);
  ok &= plan_mm(&e->mm[MM_TEXT], b.wtext, D.Vt, D.Vt, D.d, 0, b.op_z, Bp, nsm, 1, 1, Ht);
  // every step's in-projection that the tick runs, in one launch (they read only this
  // tick's z); none for the persistent depformer, which does its own
  const int din_steps = D.dep_batched ? D.nq : D.dep_steps;
  if (din_steps > 0)
    ok &= plan_mm(&e->mm[MM_DIN], b.dep_inproj, D.nq * D.dd, din_steps * D.dd, D.d, 0, b.op_z,
                  Bp, nsm);
  ok &= plan_mm(&e->mm[MM_DQKV], b.dep_wqkv, D.Ld * 3 * D.dd, 3 * D.dd, D.dd, 0, b.op_dd, Bp, nsm);
  ok &= plan_mm(&e->mm[MM_DO], b.dep_wo, D.Ld * D.dd, D.dd, D.dd, 0, b.op_do, Bp, nsm);
  ok &= plan_mm(&e->mm[MM_DGU], b.dep_wgu, D.Ld * 2 * D.Fd, D.Fd, D.dd, D.Fd, b.op_dd, Bp, nsm);
  ok &= plan_mm(&e->mm[MM_DDOWN], b.dep_wdown, D.Ld * D.dd, D.dd, D.Fd, 0, b.op_fd, Bp, nsm);
  ok &= plan_mm(&e->mm[MM_DHEAD], b.dep_heads, D.nq * D.Va, D.Va, D.dd, 0, b.op_dd, Bp, nsm);
  if (D.dep_batched) {
    const int nb = kDepBatch;
    ok &= plan_mm(&e->mm[MM_BDQKV], b.dep_wqkv, D.Ld * 3 * D.dd, 3 * D.dd, D.dd, 0, b.op_ddb, Bp,
                  nsm, nb, nb);
    ok &= plan_mm(&e->mm[MM_BDO], b.dep_wo, D.Ld * D.dd, D.dd, D.dd, 0, b.op_dob, Bp, nsm, nb, nb);
    ok &= plan_mm(&e->mm[MM_BDGU], b.dep_wgu, D.Ld * 2 * D.Fd, D.Fd, D.dd, D.Fd, b.op_ddb, Bp, nsm,
                  nb, nb);
    ok &= plan_mm(&e->mm[MM_BDDOWN], b.dep_wdown, D.Ld * D.dd, D.dd, D.Fd, 0, b.op_fdb, Bp, nsm,
                  nb, nb);
    ok &= plan_mm(&e->mm[MM_BDHEAD], b.dep_heads, D.nq * D.Va, D.Va, D.dd, 0, b.op_ddb, Bp, nsm,
                  nb, nb);
  }
  return ok;
}

// One tensor-core contraction launch: matrix `row0` rows into its stacked tensor.
// Fused RMSNorm wiring of one contraction launch: what it consumes (partials of the
// producer before it, or a stored 1/rms) and what it produces for the next one.
struct NormIO {
  const float* ssq_in = nullptr;
  int nparts = 0;
  int K = 0;
  const float* rstd_in = nullptr;
  float* rstd_out = nullptr;
  const float* alpha_out = nullptr;   // alpha of the next norm (producer)
  uint16_t* op_next = nullptr;
  float* ssq_out = nullptr;
};

// Column chunks of one launch (the batched depformer steps): strides per chunk.
struct Chunks {
  int n = 1;
  int a_rows = 0, b_rows = 0;
  long long y = 0, op = 0, emb = 0;
  int ssq_out = 0, ssq_in = 0, tok = 0;
  const int32_t* tok_ptr = nullptr;   // tokens of chunk 0 (default: b.tok)
};

cudaError_t mm_launch(const Dims& D, const Buffers& b, const Mm& g, int row0, int epi, float* Y,
                      int ldy, const uint16_t* emb, uint16_t* op_out, int ld_op, cudaStream_t s,
                      const NormIO& nio = NormIO(), const Chunks& ch = Chunks(),
                      const DecideArgs* dec = nullptr, const RopeArgs* rope = nullptr) {
  UmmaArgs a{};
  if (dec) a.dec = *dec;
  if (rope) a.rope = *rope;
  a.halves = g.H;
  a.early_trigger = D.B <= kEarlyTriggerMaxB;
  a.chunks = ch.n;
  a.a_chunk_rows = ch.a_rows;
  a.b_chunk_rows = ch.b_rows;
  a.y_chunk = ch.y;
  a.op_chunk = ch.op;
  a.ssq_out_chunk = ch.ssq_out;
  a.ssq_in_chunk = ch.ssq_in;
  a.emb_chunk = ch.emb;
  a.tok_chunk = ch.tok;
  a.ssq_in = nio.ssq_in;
  a.ssq_nparts = nio.nparts;
  a.ssq_K = nio.K;
  a.eps = D.eps;
  a.rstd_in = nio.rstd_in;
  a.rstd_out = nio.rstd_out;
  a.norm_alpha = nio.alpha_out;
  a.norm_op = nio.op_next;
  a.ssq_out = nio.ssq_out;
  a.M = g.M;
  a.pair_rows = g.pair;
  a.row0 = row0;
  a.kblocks = g.kblocks;
  a.splits = g.splits;
  a.m_tiles = g.m_tiles;
  a.B = D.B;
  a.N = 2 * D.Bp;
  a.epi = epi;
  a.Y = Y;
  a.ldy = ldy;
  a.emb = emb;
  a.tok = ch.tok_ptr ? ch.tok_ptr : b.tok;
  a.op_out = op_out;
  a.ld_op = ld_op;
  a.Bp_out = D.Bp;
  a.status = b.status;
  a.test_ctl = b.test_ctl;
  return launch_umma(a, g.mapA, g.mapB, s);
}

#define MARK(k)                                 \
  do {                                          \
    if (prof) PP_TRY(prof->mark((k), s));       \
  } while (0)

// Depformer steps 8..15 as one batched pass.  Once step 7 has decided row 8, every input
// of these steps is known (row 8, then the user codes of rows 9..15), and the layers'
// weights are shared by all steps: each contraction runs once over 8 column chunks, one
// per step (step 8 + c in chunk c), and the step attention takes all 8 at once.  Each
// chunk computes exactly what its step computes one at a time: its own in-projection
// and head, the shared layers, causal attention over steps 0..8+c of the frame.
cudaError_t enqueue_user_steps_batched(const Group* e, cudaStream_t s, Prof* prof) {
  const Dims& D = e->D;
  const Buffers& b = e->buf;
  const Mm* mm = e->mm;
  const int nb = kDepBatch, k0 = D.nq - kDepBatch;
  const int p_din = 1;   // k_dep_in: one sum of y^2 per slot and step
  const int p_do = mm[MM_BDO].m_tiles * mm[MM_BDO].splits;
  const int p_ddown = mm[MM_BDDOWN].m_tiles * mm[MM_BDDOWN].splits;
  const long long opd = 2LL * D.Bp * D.dd, opf = 2LL * D.Bp * D.Fd;
  const int R = 2 * D.Bp;
  // inputs of steps 8..15: P_{8+c} z (this tick's all-steps in-projection) + the audio
  // table 8 + c - 1 at the chunk's token
  MARK(PP_K_DEP_INPROJ);
  PP_TRY(launch_dep_in(D, b, k0, nb, b.tokb, b.dep_emb_audio + (size_t)(k0 - 1) * (D.Va + 1) * D.dd,
                       (long long)(D.Va + 1) * D.dd, b.y_b, (long long)D.B * D.dd, b.op_ddb, opd,
                       s));
  for (int j = 0; j < D.Ld; ++j) {
    NormIO qn;
    qn.ssq_in = b.ssq;
    qn.nparts = (j == 0) ? p_din : p_ddown;
    qn.K = D.dd;
    Chunks cq;
    cq.n = nb;
    cq.b_rows = R;
    cq.y = 3LL * D.B * D.dd;
    cq.ssq_in = qn.nparts * D.B;
    MARK(PP_K_DEP_QKV);
    PP_TRY(mm_launch(D, b, mm[MM_BDQKV], j * 3 * D.dd, EPI_STORE, b.dqkv_b, 3 * D.dd, nullptr,
                     nullptr, 0, s, qn, cq));
    MARK(PP_K_DEP_ATTN);
    PP_TRY(launch_dep_attn_batch(D, b, j, s));
    NormIO on;
    on.alpha_out = b.dep_mlp_alpha + (size_t)j * D.dd;
    on.op_next = b.op_ddb;
    on.ssq_out = b.ssq;
    Chunks co;
    co.n = nb;
    co.b_rows = R;
    co.y = (long long)D.B * D.dd;
    co.op = opd;
    co.ssq_out = p_do * D.B;
    MARK(PP_K_DEP_OPROJ);
    PP_TRY(mm_launch(D, b, mm[MM_BDO], j * D.dd, EPI_ADD, b.y_b, D.dd, nullptr, nullptr, 0, s, on,
                     co));
    NormIO gn;
    gn.ssq_in = b.ssq;
    gn.nparts = p_do;
    gn.K = D.dd;
    Chunks cg;
    cg.n = nb;
    cg.b_rows = R;
    cg.op = opf;
    cg.ssq_in = p_do * D.B;
    MARK(PP_K_DEP_GATEUP);
    PP_TRY(mm_launch(D, b, mm[MM_BDGU], j * 2 * D.Fd, EPI_SILU, nullptr, 0, nullptr, b.op_fdb,
                     D.Fd, s, gn, cg));
    NormIO dn;
    const bool last = (j + 1 == D.Ld);
    dn.alpha_out = last ? b.dep_out_alpha : b.dep_attn_alpha + (size_t)(j + 1) * D.dd;
    dn.op_next = b.op_ddb;
    dn.ssq_out = b.ssq;
    Chunks cd;
    cd.n = nb;
    cd.b_rows = R;
    cd.y = (long long)D.B * D.dd;
    cd.op = opd;
    cd.ssq_out = p_ddown * D.B;
    MARK(PP_K_DEP_DOWN);
    PP_TRY(mm_launch(D, b, mm[MM_BDDOWN], j * D.dd, EPI_ADD, b.y_b, D.dd, nullptr, nullptr, 0, s,
                     dn, cd));
  }
  NormIO hn;
  hn.ssq_in = b.ssq;
  hn.nparts = p_ddown;
  hn.K = D.dd;
  Chunks chd;
  chd.n = nb;
  chd.a_rows = D.Va;                       // head H_{8+c}
  chd.b_rows = R;
  chd.y = D.Va;                            // its logits follow in the same row
  chd.ssq_in = p_ddown * D.B;
  MARK(PP_K_DEP_HEAD);
  return mm_launch(D, b, mm[MM_BDHEAD], k0 * D.Va, EPI_STORE,
                   b.logits + D.Vt + (size_t)k0 * D.Va, D.logits_ld, nullptr, nullptr, 0, s, hn,
                   chd);
}

// The temporal layer `l`'s RoPE and ring append, for the qkv contraction's epilogue.
RopeArgs rope_args(const Dims& D, const Buffers& b, int l) {
  RopeArgs r{};
  r.live = b.live;
  r.pos = b.pos;
  r.cs = b.rope_cs;
  r.q = b.q;
  r.q_op = b.q_op;
  r.ring = b.ring + (size_t)l * D.B * 2 * D.H * D.W * D.Dh;
  r.d = D.d;
  r.H = D.H;
  r.Dh = D.Dh;
  r.W = D.W;
  return r;
}

// The fused greedy decision of a head launch (kind 1: text row 0; kind 2: depformer step
// `step`).
bool make_decide(const Dims& D, const Buffers& b, const Mm& g, int kind, int step,
                 DecideArgs* d) {
  (void)g;
  *d = DecideArgs{};
  d->kind = kind;
  d->step = step;
  d->V = kind == 1 ? D.Vt : D.Va;
  d->tokb = kind == 2 && D.dep_batched && step == D.dep_steps - 1;
  d->key = b.dkey + (kind == 1 ? 0 : D.B);
  d->nan = b.dnan + (kind == 1 ? 0 : 1);
  d->ticket = b.dticket + (kind == 1 ? 0 : 1);
  d->live = b.live;
  d->fmask = b.in_fmask;
  d->forced = b.in_forced;
  d->user = b.in_user;
  d->pos = b.pos;
  d->out_col = b.out_col;
  d->tok = b.tok;
  d->tok_b = b.tokb;
  d->hist = b.hist;
  d->hist_len = b.hist_len;
  d->hist_ld = kHist;
  return true;
}

// The tick with every weight contraction on the tensor cores.  RMSNorms are fused: each
// residual-producing contraction writes the next contraction's operand (alpha * y, split
// bf16) and per-slice sums of y^2; the consuming contraction scales by 1/rms.
// greedy: the greedy-only tick, whose text and depformer heads take their decisions in
// their own epilogues (no decision kernels; no sampled slot may be open)
cudaError_t enqueue_tick_tensor(const Group* e, int dep_priority, cudaStream_t s, Prof* prof,
                                bool greedy) {
  const Dims& D = e->D;
  const Buffers& b = e->buf;
  const Mm* mm = e->mm;
  // fused-norm partials: one per CTA (M-tile x split) of the producing contraction
  const int p_o = mm[MM_O].m_tiles * mm[MM_O].splits;
  const int p_down = mm[MM_DOWN].m_tiles * mm[MM_DOWN].splits;
  const int p_do = mm[MM_DO].m_tiles * mm[MM_DO].splits;
  const int p_ddown = mm[MM_DDOWN].m_tiles * mm[MM_DDOWN].splits;
  // the K-split epilogue finalises whole 4-row groups of one slot, i.e. two RoPE pairs
  const bool rope_fused = mm[MM_QKV].splits > 1;
  MARK(PP_K_BEGIN);
  PP_TRY(launch_begin(D, b, b.attn_alpha, b.op_d, b.ssq, s));
  for (int l = 0; l < D.L; ++l) {
    NormIO qn;
    qn.ssq_in = b.ssq;
    qn.nparts = (l == 0) ? 1 : p_down;
    qn.K = D.d;
    MARK(PP_K_QKV);
    if (rope_fused) {   // RoPE and the ring append in the contraction's epilogue
      RopeArgs ra = rope_args(D, b, l);
      PP_TRY(mm_launch(D, b, mm[MM_QKV], l * 3 * D.d, EPI_ROPE, nullptr, 0, nullptr, nullptr, 0,
                       s, qn, Chunks(), nullptr, &ra));
    } else {
      PP_TRY(mm_launch(D, b, mm[MM_QKV], l * 3 * D.d, EPI_STORE, b.qkv, 3 * D.d, nullptr, nullptr,
                       0, s, qn));
      MARK(PP_K_ROPE_RING);
      PP_TRY(launch_rope_ring(D, b, l, s));
    }
    MARK(PP_K_ATTN);
    PP_TRY(launch_attn(D, b, l, true, e->has_amaps ? &e->amaps : nullptr, s));
    NormIO on;
    on.alpha_out = b.mlp_alpha + (size_t)l * D.d;
    on.op_next = b.op_d;
    on.ssq_out = b.ssq;
    MARK(PP_K_OPROJ);
    PP_TRY(mm_launch(D, b, mm[MM_O], l * D.d, EPI_ADD, b.x, D.d, nullptr, nullptr, 0, s, on));
    NormIO gn;
    gn.ssq_in = b.ssq;
    gn.nparts = p_o;
    gn.K = D.d;
    MARK(PP_K_GATEUP);
    PP_TRY(mm_launch(D, b, mm[MM_GU], l * 2 * D.F, EPI_SILU, nullptr, 0, nullptr, b.op_f, D.F, s, gn));
    NormIO dn;
    const bool last = (l + 1 == D.L);
    dn.alpha_out = last ? b.out_alpha : b.attn_alpha + (size_t)(l + 1) * D.d;
    dn.op_next = last ? b.op_z : b.op_d;
    dn.ssq_out = b.ssq;
    MARK(PP_K_DOWN);
    PP_TRY(mm_launch(D, b, mm[MM_DOWN], l * D.d, EPI_ADD, b.x, D.d, nullptr, nullptr, 0, s, dn));
  }
  {
    NormIO tn;
    tn.ssq_in = b.ssq;
    tn.nparts = p_down;
    tn.K = D.d;
    tn.rstd_out = b.rstd_z;     // kept for the persistent depformer's input projections
    if (D.dep_steps > 0 || D.dep_batched) {
      // every depformer step's in-projection P_k z at once: it reads only z, so it runs
      // before the text head decides the first token; each step adds its token's row
      NormIO pn;
      pn.ssq_in = b.ssq;
      pn.nparts = p_down;
      pn.K = D.d;
      MARK(PP_K_DEP_INPROJ);
      PP_TRY(mm_launch(D, b, mm[MM_DIN], 0, EPI_STORE, b.pz, D.nq * D.dd, nullptr, nullptr, 0, s,
                       pn));
    }
    DecideArgs dt;
    const bool fuse = greedy && make_decide(D, b, mm[MM_TEXT], 1, 0, &dt);
    MARK(PP_K_TEXT_HEAD);
    PP_TRY(mm_launch(D, b, mm[MM_TEXT], 0, EPI_STORE, b.logits, D.logits_ld, nullptr, nullptr, 0, s, tn,
                     Chunks(), fuse ? &dt : nullptr));
    if (!fuse) {
      MARK(PP_K_TEXT_HEAD);
      PP_TRY(launch_text_argmax(D, b, s));
    }
  }
  if (D.dep_persist) {   // all 16 steps in one persistent kernel
    PP_TRY(cudaMemsetAsync(b.pbar, 0, 4 * sizeof(unsigned), s));   // barrier words
    PersistArgs pa;
    pa.D = D;
    pa.b = b;
    pa.bar_count = b.pbar;
    pa.bar_gen = b.pbar + 1;
    pa.abort = reinterpret_cast<int*>(b.pbar + 2);
    pa.part_val = b.ppart_val;
    pa.part_idx = b.ppart_idx;
    MARK(PP_K_DEP_PERSIST);
    PP_TRY(launch_dep_persist(pa, s));
  }
  g_launch_priority = dep_priority;   // the latency-bound depformer goes first
  for (int k = 0; k < D.dep_steps; ++k) {
    const uint16_t* emb =
        (k == 0) ? b.dep_emb_text : b.dep_emb_audio + (size_t)(k - 1) * (D.Va + 1) * D.dd;
    MARK(PP_K_DEP_INPROJ);
    PP_TRY(launch_dep_in(D, b, k, 1, b.tok, emb, 0, b.y, 0, b.op_dd, 0, s));
    for (int j = 0; j < D.Ld; ++j) {
      NormIO qn;
      qn.ssq_in = b.ssq;
      qn.nparts = (j == 0) ? 1 : p_ddown;   // k_dep_in: one partial per slot
      qn.K = D.dd;
      MARK(PP_K_DEP_QKV);
      PP_TRY(mm_launch(D, b, mm[MM_DQKV], j * 3 * D.dd, EPI_STORE, b.dqkv, 3 * D.dd, nullptr,
                       nullptr, 0, s, qn));
      MARK(PP_K_DEP_ATTN);
      PP_TRY(launch_dep_attn(D, b, k, j, true, s));
      NormIO on;
      on.alpha_out = b.dep_mlp_alpha + (size_t)j * D.dd;
      on.op_next = b.op_dd;
      on.ssq_out = b.ssq;
      MARK(PP_K_DEP_OPROJ);
      PP_TRY(mm_launch(D, b, mm[MM_DO], j * D.dd, EPI_ADD, b.y, D.dd, nullptr, nullptr, 0, s, on));
      NormIO gn;
      gn.ssq_in = b.ssq;
      gn.nparts = p_do;
      gn.K = D.dd;
      MARK(PP_K_DEP_GATEUP);
      PP_TRY(mm_launch(D, b, mm[MM_DGU], j * 2 * D.Fd, EPI_SILU, nullptr, 0, nullptr, b.op_fd,
                       D.Fd, s, gn));
      NormIO dn;
      const bool last = (j + 1 == D.Ld);
      dn.alpha_out = last ? b.dep_out_alpha : b.dep_attn_alpha + (size_t)(j + 1) * D.dd;
      dn.op_next = b.op_dd;
      dn.ssq_out = b.ssq;
      MARK(PP_K_DEP_DOWN);
      PP_TRY(mm_launch(D, b, mm[MM_DDOWN], j * D.dd, EPI_ADD, b.y, D.dd, nullptr, nullptr, 0, s, dn));
    }
    NormIO hn;
    hn.ssq_in = b.ssq;
    hn.nparts = p_ddown;
    hn.K = D.dd;
    DecideArgs dh;
    const bool fuse = greedy && make_decide(D, b, mm[MM_DHEAD], 2, k, &dh);
    MARK(PP_K_DEP_HEAD);
    PP_TRY(mm_launch(D, b, mm[MM_DHEAD], k * D.Va, EPI_STORE, b.logits + D.Vt + (size_t)k * D.Va,
                     D.logits_ld, nullptr, nullptr, 0, s, hn, Chunks(), fuse ? &dh : nullptr));
    if (!fuse) {
      MARK(PP_K_DEP_HEAD);
      PP_TRY(launch_dep_argmax(D, b, k, s));
    }
  }
  if (D.dep_batched) PP_TRY(enqueue_user_steps_batched(e, s, prof));
  if (D.dep_steps < D.nq && !D.dep_persist) {
    MARK(PP_K_DEP_HEAD);
    PP_TRY(launch_user_rows(D, b, s));
  }
  MARK(PP_K_FINISH);
  PP_TRY(launch_finish(D, b, s));
  MARK(PP_K_COUNT);
  return cudaSuccess;
}

// The tick with the CUDA-core contractions.  With prof != nullptr a timing event is
// recorded before every launch (and once at the end).
cudaError_t enqueue_tick_cc(const Dims& D, const Buffers& b, const AttnMaps* amaps, cudaStream_t s,
                            Prof* prof) {
  MARK(PP_K_BEGIN);
  PP_TRY(launch_begin(D, b, nullptr, nullptr, nullptr, s));
  for (int l = 0; l < D.L; ++l) {
    MARK(PP_K_NORM);
    PP_TRY(launch_rmsnorm(D, b.x, D.d, b.attn_alpha + (size_t)l * D.d, D.d, b.xn, D.d, nullptr, s));
    GemvArgs a{};
    a.W = b.wqkv + (size_t)l * 3 * D.d * D.d; a.M = 3 * D.d; a.K = D.d;
    a.X = b.xn; a.ldx = D.d; a.Y = b.qkv; a.ldy = 3 * D.d; a.epi = EPI_STORE;
    MARK(PP_K_QKV);
    PP_TRY(launch_gemv(D, a, s));
    MARK(PP_K_ROPE_RING);
    PP_TRY(launch_rope_ring(D, b, l, s));
    MARK(PP_K_ATTN);
    PP_TRY(launch_attn(D, b, l, false, amaps, s));
    a = GemvArgs{};
    a.W = b.wo + (size_t)l * D.d * D.d; a.M = D.d; a.K = D.d;
    a.X = b.o; a.ldx = D.d; a.Y = b.x; a.ldy = D.d; a.epi = EPI_ADD;
    MARK(PP_K_OPROJ);
    PP_TRY(launch_gemv(D, a, s));
    MARK(PP_K_NORM);
    PP_TRY(launch_rmsnorm(D, b.x, D.d, b.mlp_alpha + (size_t)l * D.d, D.d, b.xn, D.d, nullptr, s));
    a = GemvArgs{};
    a.W = b.wgu + (size_t)l * 2 * D.F * D.d; a.M = D.F; a.K = D.d;
    a.X = b.xn; a.ldx = D.d; a.Y = b.hmlp; a.ldy = D.F; a.epi = EPI_SILU;
    MARK(PP_K_GATEUP);
    PP_TRY(launch_gemv(D, a, s));
    a = GemvArgs{};
    a.W = b.wdown + (size_t)l * D.d * D.F; a.M = D.d; a.K = D.F;
    a.X = b.hmlp; a.ldx = D.F; a.Y = b.x; a.ldy = D.d; a.epi = EPI_ADD;
    MARK(PP_K_DOWN);
    PP_TRY(launch_gemv(D, a, s));
  }
  MARK(PP_K_TEXT_HEAD);
  PP_TRY(launch_rmsnorm(D, b.x, D.d, b.out_alpha, D.d, b.z, D.d, nullptr, s));
  {
    GemvArgs a{};
    a.W = b.wtext; a.M = D.Vt; a.K = D.d;
    a.X = b.z; a.ldx = D.d; a.Y = b.logits; a.ldy = D.logits_ld; a.epi = EPI_STORE;
    MARK(PP_K_TEXT_HEAD);
    PP_TRY(launch_gemv(D, a, s));
  }
  MARK(PP_K_TEXT_HEAD);
  PP_TRY(launch_text_argmax(D, b, s));
  for (int k = 0; k < D.dep_steps; ++k) {
    GemvArgs a{};
    a.W = b.dep_inproj + (size_t)k * D.dd * D.d; a.M = D.dd; a.K = D.d;
    a.X = b.z; a.ldx = D.d; a.Y = b.y; a.ldy = D.dd; a.epi = EPI_EMB;
    a.emb = (k == 0) ? b.dep_emb_text : b.dep_emb_audio + (size_t)(k - 1) * (D.Va + 1) * D.dd;
    a.tok = b.tok;
    MARK(PP_K_DEP_INPROJ);
    PP_TRY(launch_gemv(D, a, s));
    for (int j = 0; j < D.Ld; ++j) {
      MARK(PP_K_DEP_NORM);
    PP_TRY(launch_rmsnorm(D, b.y, D.dd, b.dep_attn_alpha + (size_t)j * D.dd, D.dd, b.yn, D.dd, nullptr, s));
      a = GemvArgs{};
      a.W = b.dep_wqkv + (size_t)j * 3 * D.dd * D.dd; a.M = 3 * D.dd; a.K = D.dd;
      a.X = b.yn; a.ldx = D.dd; a.Y = b.dqkv; a.ldy = 3 * D.dd; a.epi = EPI_STORE;
      MARK(PP_K_DEP_QKV);
    PP_TRY(launch_gemv(D, a, s));
      MARK(PP_K_DEP_ATTN);
    PP_TRY(launch_dep_attn(D, b, k, j, false, s));
      a = GemvArgs{};
      a.W = b.dep_wo + (size_t)j * D.dd * D.dd; a.M = D.dd; a.K = D.dd;
      a.X = b.dout; a.ldx = D.dd; a.Y = b.y; a.ldy = D.dd; a.epi = EPI_ADD;
      MARK(PP_K_DEP_OPROJ);
    PP_TRY(launch_gemv(D, a, s));
      MARK(PP_K_DEP_NORM);
    PP_TRY(launch_rmsnorm(D, b.y, D.dd, b.dep_mlp_alpha + (size_t)j * D.dd, D.dd, b.yn, D.dd, nullptr, s));
      a = GemvArgs{};
      a.W = b.dep_wgu + (size_t)j * 2 * D.Fd * D.dd; a.M = D.Fd; a.K = D.dd;
      a.X = b.yn; a.ldx = D.dd; a.Y = b.dh; a.ldy = D.Fd; a.epi = EPI_SILU;
      MARK(PP_K_DEP_GATEUP);
    PP_TRY(launch_gemv(D, a, s));
      a = GemvArgs{};
      a.W = b.dep_wdown + (size_t)j * D.dd * D.Fd; a.M = D.dd; a.K = D.Fd;
      a.X = b.dh; a.ldx = D.Fd; a.Y = b.y; a.ldy = D.dd; a.epi = EPI_ADD;
      MARK(PP_K_DEP_DOWN);
    PP_TRY(launch_gemv(D, a, s));
    }
    MARK(PP_K_DEP_NORM);
    PP_TRY(launch_rmsnorm(D, b.y, D.dd, b.dep_out_alpha, D.dd, b.yn, D.dd, nullptr, s));
    a = GemvArgs{};
    a.W = b.dep_heads + (size_t)k * D.Va * D.dd; a.M = D.Va; a.K = D.dd;
    a.X = b.yn; a.ldx = D.dd; a.Y = b.logits + D.Vt + (size_t)k * D.Va; a.ldy = D.logits_ld;
    a.epi = EPI_STORE;
    MARK(PP_K_DEP_HEAD);
    PP_TRY(launch_gemv(D, a, s));
    MARK(PP_K_DEP_HEAD);
    PP_TRY(launch_dep_argmax(D, b, k, s));
  }
  if (D.dep_steps < D.nq) {
    MARK(PP_K_DEP_HEAD);
    PP_TRY(launch_user_rows(D, b, s));
  }
  MARK(PP_K_FINISH);
  PP_TRY(launch_finish(D, b, s));
  MARK(PP_K_COUNT);   // end marker
  return cudaSuccess;
}

cudaError_t enqueue_group(const pp_engine* e, int g, cudaStream_t s, Prof* prof, bool greedy) {
  g_launch_priority = 0;
  cudaError_t err = e->tensor ? enqueue_tick_tensor(&e->grp[g], e->dep_priority, s, prof, greedy)
                              : enqueue_tick_cc(e->grp[g].D, e->grp[g].buf,
                                                e->grp[g].has_amaps ? &e->grp[g].amaps : nullptr,
                                                s, prof);
  g_launch_priority = 0;
  return err;
}

// The whole tick: one branch per slot group (a fork/join inside the captured graph);
// the profiling graph runs the groups one after the other so that its events time
// single kernels.
cudaError_t enqueue_tick(const pp_engine* e, cudaStream_t s, Prof* prof, bool greedy) {
  if (e->ngroups == 1 || prof) {
    for (int g = 0; g < e->ngroups; ++g) PP_TRY(enqueue_group(e, g, s, prof, greedy));
    return cudaSuccess;
  }
  PP_TRY(cudaEventRecord(e->fork, s));
  for (int g = 0; g < e->ngroups; ++g) {
    PP_TRY(cudaStreamWaitEvent(e->branch[g], e->fork, 0));
    PP_TRY(enqueue_group(e, g, e->branch[g], nullptr, greedy));
    PP_TRY(cudaEventRecord(e->join[g], e->branch[g]));
    PP_TRY(cudaStreamWaitEvent(s, e->join[g], 0));
  }
  return cudaSuccess;
}

int weight_dims(const pp_config* c, int which, int64_t d[4], int* nd, int* f32) {
  const int64_t dm = c->d_model, L = c->n_layers, F = c->ffn, Vt = c->text_vocab,
                Va = c->audio_card, nq = c->n_q, dd = c->dep_d, Ld = c->dep_layers,
                Fd = c->dep_ffn;
  *f32 = 0;
  auto set = [&](int n, int64_t a, int64_t b2, int64_t c2) {
    *nd = n; d[0] = a; d[1] = b2; d[2] = c2; d[3] = 0;
  };
  switch (which) {
    case PP_W_EMB_TEXT: set(2, Vt + 1, dm, 0); break;
    case PP_W_EMB_AUDIO: set(3, nq, Va + 1, dm); break;
    case PP_W_ATTN_ALPHA: set(2, L, dm, 0); *f32 = 1; break;
    case PP_W_QKV: set(3, L, 3 * dm, dm); break;
    case PP_W_O: set(3, L, dm, dm); break;
    case PP_W_MLP_ALPHA: set(2, L, dm, 0); *f32 = 1; break;
    case PP_W_GU: set(3, L, 2 * F, dm); break;
    case PP_W_DOWN: set(3, L, dm, F); break;
    case PP_W_OUT_ALPHA: set(1, dm, 0, 0); *f32 = 1; break;
    case PP_W_TEXT: set(2, Vt, dm, 0); break;
    case PP_W_DEP_INPROJ: set(3, nq, dd, dm); break;
    case PP_W_DEP_EMB_TEXT: set(2, Vt + 1, dd, 0); break;
    case PP_W_DEP_EMB_AUDIO: set(3, nq - 1, Va + 1, dd); break;
    case PP_W_DEP_ATTN_ALPHA: set(2, Ld, dd, 0); *f32 = 1; break;
    case PP_W_DEP_QKV: set(3, Ld, 3 * dd, dd); break;
    case PP_W_DEP_O: set(3, Ld, dd, dd); break;
    case PP_W_DEP_MLP_ALPHA: set(2, Ld, dd, 0); *f32 = 1; break;
    case PP_W_DEP_GU: set(3, Ld, 2 * Fd, dd); break;
    case PP_W_DEP_DOWN: set(3, Ld, dd, Fd); break;
    case PP_W_DEP_OUT_ALPHA: set(1, dd, 0, 0); *f32 = 1; break;
    case PP_W_DEP_HEADS: set(3, nq, Va, dd); break;
    default: return PP_EINVAL;
  }
  return PP_OK;
}

}  // namespace

extern "C" {

int pp_weight_shape(const pp_config* c, int which, int64_t dims[4], int* ndim, int* is_f32) {
  if (!config_ok(c) || !dims || !ndim || !is_f32) return PP_EINVAL;
  return weight_dims(c, which, dims, ndim, is_f32);
}

size_t pp_workspace_bytes(const pp_config* c) {
  if (!config_ok(c)) return 0;
  return carve(c, nullptr, nullptr, nullptr);
}

int pp_create(const pp_config* c, const pp_weights* w, void* workspace, size_t ws_bytes,
              pp_engine** out) {
  if (!out) return PP_EINVAL;
  *out = nullptr;
  if (!config_ok(c) || !w || !workspace) return PP_EINVAL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return PP_EINVAL;
  for (int i = 0; i < PP_W_COUNT; ++i)
    if (!w->ptr[i] || (reinterpret_cast<uintptr_t>(w->ptr[i]) & 15)) return PP_EINVAL;
  pp_engine* e = new (std::nothrow) pp_engine();
  if (!e) return PP_EINVAL;
  const size_t need = carve(c, reinterpret_cast<char*>(workspace), &e->shared, e->grp);
  if (ws_bytes < need) {
    delete e;
    return PP_E_NOSPACE;
  }
  e->cfg = *c;
  e->B = c->max_batch;
  e->ngroups = group_count(c);
  e->logits_ld = c->text_vocab + c->n_q * c->audio_card;
  for (int g = 0; g < e->ngroups; ++g) {
    Buffers& b = e->grp[g].buf;
    b.emb_text = (const uint16_t*)w->ptr[PP_W_EMB_TEXT];
    b.emb_audio = (const uint16_t*)w->ptr[PP_W_EMB_AUDIO];
    b.attn_alpha = (const float*)w->ptr[PP_W_ATTN_ALPHA];
    b.wqkv = (const uint16_t*)w->ptr[PP_W_QKV];
    b.wo = (const uint16_t*)w->ptr[PP_W_O];
    b.mlp_alpha = (const float*)w->ptr[PP_W_MLP_ALPHA];
    b.wgu = (const uint16_t*)w->ptr[PP_W_GU];
    b.wdown = (const uint16_t*)w->ptr[PP_W_DOWN];
    b.out_alpha = (const float*)w->ptr[PP_W_OUT_ALPHA];
    b.wtext = (const uint16_t*)w->ptr[PP_W_TEXT];
    b.dep_inproj = (const uint16_t*)w->ptr[PP_W_DEP_INPROJ];
    b.dep_emb_text = (const uint16_t*)w->ptr[PP_W_DEP_EMB_TEXT];
    b.dep_emb_audio = (const uint16_t*)w->ptr[PP_W_DEP_EMB_AUDIO];
    b.dep_attn_alpha = (const float*)w->ptr[PP_W_DEP_ATTN_ALPHA];
    b.dep_wqkv = (const uint16_t*)w->ptr[PP_W_DEP_QKV];
    b.dep_wo = (const uint16_t*)w->ptr[PP_W_DEP_O];
    b.dep_mlp_alpha = (const float*)w->ptr[PP_W_DEP_MLP_ALPHA];
    b.dep_wgu = (const uint16_t*)w->ptr[PP_W_DEP_GU];
    b.dep_wdown = (const uint16_t*)w->ptr[PP_W_DEP_DOWN];
    b.dep_out_alpha = (const float*)w->ptr[PP_W_DEP_OUT_ALPHA];
    b.dep_heads = (const uint16_t*)w->ptr[PP_W_DEP_HEADS];
  }
  e->ctl.assign(e->B, 0);
  e->ctl_pos.assign(e->B, 0);
  e->pos.assign(e->B, 0);
  e->open.assign(e->B, 0);
  e->samp.assign(e->B, SampleParams{});

  e->tensor = !(c->flags & PP_FLAG_CUDA_CORE_GEMM);
  g_use_pdl = !(c->flags & PP_FLAG_NO_PDL);   // read while this engine's graphs are captured
  cudaError_t err = cudaSuccess;
  {  // zero the per-slot state (positions, liveness, control, status, sampling, history)
    const Buffers& sh = e->shared;
    err = cudaMemset(sh.pos, 0, (size_t)(reinterpret_cast<char*>(sh.in_col) -
                                          reinterpret_cast<char*>(sh.pos)));
  }
  for (int g = 0; g < e->ngroups && err == cudaSuccess; ++g) {
    const Buffers& b = e->grp[g].buf;
    const Dims& D = e->grp[g].D;
    err = cudaMemset(b.attn_count, 0, sizeof(uint32_t) * (size_t)D.B * D.H);
    if (err == cudaSuccess) {   // operands: their padding rows stay zero
      char* op_lo = reinterpret_cast<char*>(b.op_d);
      char* op_hi = reinterpret_cast<char*>(b.op_fdb + (size_t)kDepBatch * 2 * D.Bp * D.Fd);
      err = cudaMemset(op_lo, 0, (size_t)(op_hi - op_lo));
    }
  }
  for (int g = 0; g < e->ngroups && err == cudaSuccess; ++g) {
    Group* gr = &e->grp[g];
    const Dims& D = gr->D;
    if (D.Dh == 128) {   // the tensor-core attention reads the ring through tensor maps
      const size_t blk = (size_t)D.H * D.W * D.Dh;
      gr->has_amaps = attn_maps(&gr->amaps, gr->buf.ring, gr->buf.ring + blk, 2 * blk, D.L * D.B,
                                D.H, D.W, D.Dh, gr->buf.q_op, D.B * D.H);
      if (!gr->has_amaps) err = cudaErrorInvalidValue;
    }
  }
  for (int g = 0; g < e->ngroups && err == cudaSuccess; ++g) {
    err = sample_setup(e->grp[g].D);
    if (err == cudaSuccess && e->grp[g].D.dep_persist) err = persist_setup(e->grp[g].D);
  }
  if (err == cudaSuccess && e->tensor) {
    int dev = 0, nsm = 0;
    err = cudaGetDevice(&dev);
    if (err == cudaSuccess)
      err = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    for (int g = 0; g < e->ngroups && err == cudaSuccess; ++g) {
      e->grp[g].wide_tiles = (c->flags & PP_FLAG_WIDE_TILES) != 0;
      err = umma_setup(2 * e->grp[g].D.Bp);
      if (err == cudaSuccess && !plan_all(&e->grp[g], nsm)) err = cudaErrorInvalidValue;
    }
  }
  if (err == cudaSuccess && e->ngroups > 1) {
    int least = 0, greatest = 0;
    err = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    e->dep_priority = greatest;
    for (int g = 0; g < e->ngroups && err == cudaSuccess; ++g) {
      err = cudaStreamCreateWithFlags(&e->branch[g], cudaStreamNonBlocking);
      if (err == cudaSuccess) err = cudaEventCreateWithFlags(&e->join[g], cudaEventDisableTiming);
    }
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&e->fork, cudaEventDisableTiming);
  }
  if (err == cudaSuccess) err = cudaStreamCreateWithFlags(&e->cap_stream, cudaStreamNonBlocking);
  e->pdl = g_use_pdl;
  if (err == cudaSuccess)
    err = cudaStreamBeginCapture(e->cap_stream, cudaStreamCaptureModeThreadLocal);
  if (err == cudaSuccess) {
    cudaError_t le = enqueue_tick(e, e->cap_stream, nullptr, false);
    err = cudaStreamEndCapture(e->cap_stream, &e->graph);
    if (le != cudaSuccess) err = le;
  }
  if (err == cudaSuccess) err = cudaGraphInstantiate(&e->exec, e->graph, 0);
  // the greedy-only tick (the decisions fused into the heads), used while no open slot
  // samples
  if (err == cudaSuccess)
    err = cudaStreamBeginCapture(e->cap_stream, cudaStreamCaptureModeThreadLocal);
  if (err == cudaSuccess) {
    cudaError_t le = enqueue_tick(e, e->cap_stream, nullptr, true);
    err = cudaStreamEndCapture(e->cap_stream, &e->graph_greedy);
    if (le != cudaSuccess) err = le;
  }
  if (err == cudaSuccess) err = cudaGraphInstantiate(&e->exec_greedy, e->graph_greedy, 0);
  if (err == cudaSuccess) {
    size_t n = 0;
    err = cudaGraphGetNodes(e->graph_greedy, nullptr, &n);
    e->n_kernels = (int)n;
  }
  if (err == cudaSuccess) err = cudaDeviceSynchronize();
  if (err != cudaSuccess) {
    pp_destroy(e);
    return PP_E_CUDA;
  }
  *out = e;
  return PP_OK;
}

void pp_destroy(pp_engine* e) {
  if (!e) return;
  if (e->prof_exec) cudaGraphExecDestroy(e->prof_exec);
  if (e->prof_graph) cudaGraphDestroy(e->prof_graph);
  e->prof.clear();
  if (e->exec) cudaGraphExecDestroy(e->exec);
  if (e->graph) cudaGraphDestroy(e->graph);
  if (e->exec_greedy) cudaGraphExecDestroy(e->exec_greedy);
  if (e->graph_greedy) cudaGraphDestroy(e->graph_greedy);
  if (e->cap_stream) cudaStreamDestroy(e->cap_stream);
  for (int g = 0; g < kMaxGroups; ++g) {
    if (e->branch[g]) cudaStreamDestroy(e->branch[g]);
    if (e->join[g]) cudaEventDestroy(e->join[g]);
  }
  if (e->fork) cudaEventDestroy(e->fork);
  delete e;
}

static int open_at(pp_engine* e, int slot, int64_t pos) {
  if (!e) return PP_EINVAL;
  if (slot < 0 || slot >= e->B) return PP_E_RANGE;
  if (pos < 0 || pos >= 0x7FFFFFFF) return PP_E_RANGE;
  if (e->open[slot]) return PP_E_BUSY;
  e->open[slot] = 1;
  e->ctl[slot] = 1 | 2;
  e->ctl_pos[slot] = (int32_t)pos;
  e->ctl_dirty = true;
  e->pos[slot] = pos;
  e->samp[slot] = SampleParams{};   // a new session starts greedy
  e->samp_dirty = true;
  return PP_OK;
}

int pp_session_open(pp_engine* e, int slot) { return open_at(e, slot, 0); }

int pp_session_import(pp_engine* e, int slot, int64_t pos) { return open_at(e, slot, pos); }

int pp_session_close(pp_engine* e, int slot) {
  if (!e) return PP_EINVAL;
  if (slot < 0 || slot >= e->B) return PP_E_RANGE;
  if (!e->open[slot]) return PP_E_NOTLIVE;
  e->open[slot] = 0;
  e->ctl[slot] = 0;
  e->ctl_dirty = true;
  e->samp[slot] = SampleParams{};
  e->samp_dirty = true;
  return PP_OK;
}

int pp_session_sampling(pp_engine* e, int slot, const pp_sampling* p) {
  if (!e) return PP_EINVAL;
  if (slot < 0 || slot >= e->B) return PP_E_RANGE;
  if (!e->open[slot]) return PP_E_NOTLIVE;
  SampleParams sp{};
  if (p) {
    const float fs[] = {p->text_temperature, p->text_top_p, p->repetition_penalty,
                        p->audio_temperature, p->audio_top_p};
    for (float f : fs)
      if (!std::isfinite(f)) return PP_EINVAL;
    if (!(p->text_top_p > 0.f && p->text_top_p <= 1.f)) return PP_EINVAL;
    if (!(p->audio_top_p > 0.f && p->audio_top_p <= 1.f)) return PP_EINVAL;
    if (!(p->repetition_penalty > 0.f)) return PP_EINVAL;
    if (p->penalty_window < 0 || p->penalty_window > kHist) return PP_EINVAL;
    const Dims& D = e->grp[0].D;
    if (p->text_temperature > 0.f && !D.samp_text) return PP_EINVAL;
    if (p->audio_temperature > 0.f && (!D.samp_audio || D.dep_persist)) return PP_EINVAL;
    sp.t_temp = p->text_temperature;
    sp.t_top_k = p->text_top_k;
    sp.t_top_p = p->text_top_p;
    sp.penalty = p->repetition_penalty;
    sp.window = p->penalty_window;
    sp.a_temp = p->audio_temperature;
    sp.a_top_k = p->audio_top_k;
    sp.a_top_p = p->audio_top_p;
    sp.seed_lo = (uint32_t)p->seed;
    sp.seed_hi = (uint32_t)(p->seed >> 32);
  }
  e->samp[slot] = sp;
  e->samp_dirty = true;
  return PP_OK;
}

int pp_session_pos(pp_engine* e, int slot, int64_t* pos) {
  if (!e || !pos) return PP_EINVAL;
  if (slot < 0 || slot >= e->B) return PP_E_RANGE;
  if (!e->open[slot]) return PP_E_NOTLIVE;
  *pos = e->pos[slot];
  return PP_OK;
}

int pp_ring_block(pp_engine* e, int layer, int slot, int kv, void** ptr) {
  if (!e || !ptr || (kv != 0 && kv != 1)) return PP_EINVAL;
  if (layer < 0 || layer >= e->grp[0].D.L || slot < 0 || slot >= e->B) return PP_E_RANGE;
  int g = e->ngroups - 1;
  while (slot < e->grp[g].slot0) --g;
  const Dims& D = e->grp[g].D;
  const int s = slot - e->grp[g].slot0;
  *ptr = e->grp[g].buf.ring + ((((size_t)layer * D.B + s) * 2 + kv) * D.H) * (size_t)D.W * D.Dh;
  return PP_OK;
}

// True when an open slot samples a row: the tick then needs the decision kernels.
static bool any_sampling(const pp_engine* e) {
  for (int i = 0; i < e->B; ++i)
    if (e->open[i] && (e->samp[i].t_temp > 0.f || e->samp[i].a_temp > 0.f)) return true;
  return false;
}

static int step_impl(pp_engine* e, const int32_t* prev_column, const int32_t* user_codes,
                     const uint8_t* force_mask, const int32_t* forced_tokens, int32_t* column,
                     float* logits, cudaStream_t s, bool wait, cudaGraphExec_t exec) {
  if (!e || !prev_column || !user_codes || !column) return PP_EINVAL;
  if ((force_mask != nullptr) != (forced_tokens != nullptr)) return PP_EINVAL;
  const Buffers& b = e->shared;
  const size_t B = e->B;
  cudaError_t err = cudaMemcpyAsync(b.in_col, prev_column, B * kRows * 4, cudaMemcpyDefault, s);
  if (err == cudaSuccess)
    err = cudaMemcpyAsync(b.in_user, user_codes, B * PP_USER_ROWS * 4, cudaMemcpyDefault, s);
  if (err == cudaSuccess) {
    if (force_mask) {
      err = cudaMemcpyAsync(b.in_fmask, force_mask, B * kRows, cudaMemcpyDefault, s);
      if (err == cudaSuccess)
        err = cudaMemcpyAsync(b.in_forced, forced_tokens, B * kRows * 4, cudaMemcpyDefault, s);
    } else {
      err = cudaMemsetAsync(b.in_fmask, 0, B * kRows, s);
    }
  }
  // control words, only after an open/close: pageable host memory is staged by the
  // runtime before the call returns, so the host copy may change right after
  const bool upload = e->ctl_dirty;
  if (err == cudaSuccess && upload)
    err = cudaMemcpyAsync(b.ctl, e->ctl.data(), B * 4, cudaMemcpyHostToDevice, s);
  if (err == cudaSuccess && upload)
    err = cudaMemcpyAsync(b.ctl_pos, e->ctl_pos.data(), B * 4, cudaMemcpyHostToDevice, s);
  const bool upload_samp = e->samp_dirty;
  if (err == cudaSuccess && upload_samp)
    err = cudaMemcpyAsync(b.samp, e->samp.data(), B * sizeof(SampleParams), cudaMemcpyHostToDevice,
                          s);
  if (err == cudaSuccess) err = cudaGraphLaunch(exec, s);
  if (err == cudaSuccess)
    err = cudaMemcpyAsync(column, b.out_col, B * kRows * 4, cudaMemcpyDefault, s);
  if (err == cudaSuccess && logits)
    err = cudaMemcpyAsync(logits, b.logits, B * (size_t)e->logits_ld * 4, cudaMemcpyDefault, s);
  if (err == cudaSuccess && wait) err = cudaStreamSynchronize(s);
  if (err != cudaSuccess) return PP_E_CUDA;
  if (upload) {
    for (size_t i = 0; i < B; ++i) e->ctl[i] &= 1;   // the device applies a reset once
    e->ctl_dirty = false;
  }
  if (upload_samp) e->samp_dirty = false;
  for (size_t i = 0; i < B; ++i)
    if (e->open[i]) e->pos[i] += 1;
  return PP_OK;
}

int pp_step(pp_engine* e, const int32_t* prev_column, const int32_t* user_codes,
            const uint8_t* force_mask, const int32_t* forced_tokens, int32_t* column,
            float* logits, void* stream) {
  if (!e) return PP_EINVAL;
  return step_impl(e, prev_column, user_codes, force_mask, forced_tokens, column, logits,
                   (cudaStream_t)stream, false, any_sampling(e) ? e->exec : e->exec_greedy);
}

int pp_step_host(pp_engine* e, const int32_t* prev_column, const int32_t* user_codes,
                 const uint8_t* force_mask, const int32_t* forced_tokens, int32_t* column,
                 float* logits, void* stream) {
  if (!e) return PP_EINVAL;
  return step_impl(e, prev_column, user_codes, force_mask, forced_tokens, column, logits,
                   (cudaStream_t)stream, true, any_sampling(e) ? e->exec : e->exec_greedy);
}

int pp_profile_step(pp_engine* e, const int32_t* prev_column, const int32_t* user_codes,
                    const uint8_t* force_mask, const int32_t* forced_tokens, int32_t* column,
                    float* logits, void* stream, double* kind_ms, int64_t* kind_launches) {
  if (!e || !kind_ms || !kind_launches) return PP_EINVAL;
  if (!e->prof_exec) {   // capture the profiling graph on first use
    g_use_pdl = e->pdl;
    cudaError_t err = cudaStreamBeginCapture(e->cap_stream, cudaStreamCaptureModeThreadLocal);
    if (err == cudaSuccess) {
      cudaError_t le = enqueue_tick(e, e->cap_stream, &e->prof, !any_sampling(e));
      err = cudaStreamEndCapture(e->cap_stream, &e->prof_graph);
      if (le != cudaSuccess) err = le;
    }
    if (err == cudaSuccess) err = cudaGraphInstantiate(&e->prof_exec, e->prof_graph, 0);
    if (err != cudaSuccess) {
      if (e->prof_graph) cudaGraphDestroy(e->prof_graph);
      e->prof_graph = nullptr;
      e->prof.clear();
      return PP_E_CUDA;
    }
  }
  int rc = step_impl(e, prev_column, user_codes, force_mask, forced_tokens, column, logits,
                     (cudaStream_t)stream, true, e->prof_exec);
  if (rc != PP_OK) return rc;
  const size_t n = e->prof.ev.size();
  for (size_t i = 0; i + 1 < n; ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, e->prof.ev[i], e->prof.ev[i + 1]) != cudaSuccess)
      return PP_E_CUDA;
    const int k = e->prof.kind[i];
    if (k >= 0 && k < PP_K_COUNT) {
      kind_ms[k] += ms;
      kind_launches[k] += 1;
    }
  }
  return PP_OK;
}

int pp_status(pp_engine* e, void* stream, uint32_t* bits) {
  if (!e || !bits) return PP_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t v = 0;
  cudaError_t err = cudaStreamSynchronize(s);
  if (err == cudaSuccess) err = cudaMemcpy(&v, e->shared.status, 4, cudaMemcpyDeviceToHost);
  if (err == cudaSuccess) err = cudaMemset(e->shared.status, 0, 4);
  if (err == cudaSuccess) err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return PP_E_CUDA;
  *bits = v;
  return PP_OK;
}

int pp_step_kernel_count(pp_engine* e) { return e ? e->n_kernels : PP_EINVAL; }

int pp_test_faults(pp_engine* e, int32_t wait_polls, int32_t withhold, int32_t kinds,
                   void* stream) {
  if (!e || wait_polls < 0 || withhold < 0) return PP_EINVAL;
  if (kinds & ~(PP_TEST_UMMA | PP_TEST_ATTN | PP_TEST_PERSIST)) return PP_EINVAL;
  e->test_word[0] = wait_polls;
  e->test_word[1] = withhold;
  e->test_word[2] = kinds;
  e->test_word[3] = 0;
  // pageable source: the runtime stages it before returning, so the word may change next
  const cudaError_t err = cudaMemcpyAsync(e->shared.test_ctl, e->test_word, sizeof(e->test_word),
                                          cudaMemcpyHostToDevice, (cudaStream_t)stream);
  return err == cudaSuccess ? PP_OK : PP_E_CUDA;
}

int pp_sample(const float* logits, int64_t ld, int rows, int n, float temperature, int top_k,
              float top_p, float penalty, const int32_t* hist, int hist_ld,
              const int32_t* hist_n, const float* uniforms, int32_t* tokens, uint32_t* status,
              void* stream) {
  if (rows < 0 || n < 1 || ld < n || (int64_t)n * 4 > kSampleSmemMax) return PP_EINVAL;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return PP_EINVAL;
  if (!(top_p > 0.f && top_p <= 1.f) || !(penalty > 0.f) || !std::isfinite(penalty))
    return PP_EINVAL;
  if (hist && (!hist_n || hist_ld < 1 || hist_ld > kHist)) return PP_EINVAL;
  if (rows == 0) return PP_OK;
  if (!logits || !uniforms || !tokens) return PP_EINVAL;
  if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(uniforms) |
       reinterpret_cast<uintptr_t>(tokens)) & 3)
    return PP_EINVAL;
  const cudaError_t err =
      launch_sample_rows(logits, ld, rows, n, temperature, top_k, top_p, penalty, hist, hist_ld,
                         hist_n, uniforms, tokens, status, (cudaStream_t)stream);
  return err == cudaSuccess ? PP_OK : PP_E_CUDA;
}

static bool ring_attention_args_ok(int B, int H, int head_dim, int window) {
  return B >= 1 && H >= 1 && window >= 1 && head_dim_ok(head_dim) &&
         (int64_t)B * H <= (int64_t)1 << 24 && window <= (1 << 24);
}

static size_t ring_attention_part_bytes(int B, int H, int head_dim, int window) {
  const size_t nc = (size_t)(window + kAttnChunk - 1) / kAttnChunk;
  return (((size_t)B * H * attn_pair_floats((int)nc, head_dim) * sizeof(float)) + 255) &
         ~(size_t)255;
}

static size_t ring_attention_count_bytes(int B, int H) {
  return ((size_t)B * H * sizeof(uint32_t) + 255) & ~(size_t)255;
}

size_t pp_ring_attention_scratch_bytes(int B, int H, int head_dim, int window) {
  if (!ring_attention_args_ok(B, H, head_dim, window)) return 0;
  // partials | tickets | (head dim 128) the bf16 hi/lo query operand
  const size_t qop = head_dim == 128 ? (size_t)B * H * 2 * head_dim * sizeof(uint16_t) : 0;
  return ring_attention_part_bytes(B, H, head_dim, window) + ring_attention_count_bytes(B, H) +
         qop;
}

int pp_ring_attention(const float* q, const uint16_t* k, const uint16_t* v, int64_t slot_stride,
                      const int32_t* n_valid, int B, int H, int head_dim, int window,
                      float* out, uint32_t* status, void* scratch, size_t scratch_bytes,
                      void* stream) {
  if (!ring_attention_args_ok(B, H, head_dim, window)) return PP_EINVAL;
  if (!q || !k || !v || !n_valid || !out || !scratch || slot_stride < 0) return PP_EINVAL;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v)) & 15)
    return PP_EINVAL;
  if ((slot_stride & 7) || (reinterpret_cast<uintptr_t>(scratch) & 255)) return PP_EINVAL;
  if (scratch_bytes < pp_ring_attention_scratch_bytes(B, H, head_dim, window)) return PP_E_NOSPACE;
  AttnArgs a{};
  a.q = q;
  a.q_ld = H * head_dim;
  a.q_scale = 1.4426950408889634f / sqrtf((float)head_dim);
  a.k = k;
  a.v = v;
  a.slot_stride = (size_t)slot_stride;
  a.n_valid = n_valid;
  a.H = H;
  a.W = window;
  a.nc_max = (window + kAttnChunk - 1) / kAttnChunk;
  a.out = out;
  a.out_ld = H * head_dim;
  a.op = nullptr;
  a.status = status;
  char* sp = reinterpret_cast<char*>(scratch);
  a.part = reinterpret_cast<float*>(sp);
  sp += ring_attention_part_bytes(B, H, head_dim, window);
  a.count = reinterpret_cast<uint32_t*>(sp);
  sp += ring_attention_count_bytes(B, H);
  AttnMaps maps;
  if (head_dim == 128) {
    a.q_op = reinterpret_cast<uint16_t*>(sp);
    if (!attn_maps(&maps, k, v, (size_t)slot_stride, B, H, window, head_dim, a.q_op, B * H))
      return PP_EINVAL;
  }
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t err = cudaMemsetAsync(a.count, 0, (size_t)B * H * sizeof(uint32_t), s);
  if (err == cudaSuccess && head_dim == 128) err = launch_q_split(a, B, head_dim, s);
  if (err == cudaSuccess) err = launch_attn_args(a, B, head_dim, &maps, 0, s);
  return err == cudaSuccess ? PP_OK : PP_E_CUDA;
}

}  // extern "C"
