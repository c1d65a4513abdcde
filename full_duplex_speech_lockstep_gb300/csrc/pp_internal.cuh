// pp_internal.cuh - engine layout and kernel launchers of the lockstep tick (sm_103a).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pp.h"

namespace pp {

constexpr int kRows = PP_ROWS;
constexpr int kAttnChunk = 128;     // ring positions per attention work unit (split-K unit)

// Chunk partial of the ring attention: [max, sum, 0 x 6, o[Dh]] floats, so that every
// 32-byte sector is written whole; the records of one (slot, head) form a block padded
// to 128 bytes (whole L2 lines, discarded once merged).
__host__ __device__ constexpr int attn_rec_floats(int Dh) { return Dh + 8; }
__host__ __device__ constexpr size_t attn_pair_floats(int nc_max, int Dh) {
  return ((size_t)nc_max * (size_t)(Dh + 8) + 31) & ~(size_t)31;
}
constexpr int kMaxBatch = 64;

// Device-side pointers and sizes every kernel of the tick needs.
struct Dims {
  int d, L, H, Dh, F, Vt, Va, nq, dd, Ld, Hd, Dhd, Fd, W, B;
  float eps, rope_base;
  int nc_max;            // attention chunks per (slot, head) at a full ring
  int logits_ld;         // Vt + nq * Va
  int Bp;                // slots padded to a multiple of 8: operand rows are [hi: Bp][lo: Bp]
  int dep_steps;         // depformer steps run one at a time (n_q, or n_q / 2 when the
                         // user steps are elided or run as one batched pass)
  int dep_batched;       // 1: steps n_q/2 .. n_q-1 run as one batched pass
  int dep_persist;       // 1: all depformer steps run as one persistent kernel
  int samp_text;         // 1: the text decision kernel holds a logit row in shared memory
  int samp_audio;        // 1: the same for the agent audio rows
};

struct Buffers {
  // weights
  const uint16_t* emb_text;
  const uint16_t* emb_audio;
  const float* attn_alpha;
  const uint16_t* wqkv;
  const uint16_t* wo;
  const float* mlp_alpha;
  const uint16_t* wgu;
  const uint16_t* wdown;
  const float* out_alpha;
  const uint16_t* wtext;
  const uint16_t* dep_inproj;
  const uint16_t* dep_emb_text;
  const uint16_t* dep_emb_audio;
  const float* dep_attn_alpha;
  const uint16_t* dep_wqkv;
  const uint16_t* dep_wo;
  const float* dep_mlp_alpha;
  const uint16_t* dep_wgu;
  const uint16_t* dep_wdown;
  const float* dep_out_alpha;
  const uint16_t* dep_heads;
  // state
  uint16_t* ring;          // [L][B][2][H][W][Dh] bf16
  int32_t* pos;            // [B]
  int32_t* live;           // [B]
  int32_t* nvalid;         // [B] valid ring positions this tick (0 = closed slot)
  int32_t* ctl;            // [B] host-uploaded control: bit0 live, bit1 reset position
  int32_t* ctl_pos;        // [B] position applied when bit1 is set
  uint32_t* status;        // [1]
  int32_t* test_ctl;       // [4] fault-test word (pp_test_faults): poll budget, copies to
                           // withhold, kernel families; zeros in normal operation
  struct SampleParams* samp;   // [B] sampling parameters (greedy when temperature <= 0)
  int32_t* hist_len;       // [B] text tokens recorded since open (capped at kHist)
  int32_t* hist;           // [B][kHist] text token of position p at p mod kHist
  // per-tick inputs / outputs (staged)
  int32_t* in_col;         // [B][17]
  int32_t* in_user;        // [B][8]
  uint8_t* in_fmask;       // [B][17]
  int32_t* in_forced;      // [B][17]
  int32_t* out_col;        // [B][17]
  // activations and scratch
  float* x;                // [B][d]
  float* xn;               // [B][max(d, F)] normalised input of the next contraction
  float* z;                // [B][d] post final norm (text head and depformer input)
  float* qkv;              // [B][3d]
  float* q;                // [B][d] rotated, pre-scaled query
  uint16_t* q_op;          // [B][H][2][Dh] the same query as bf16 hi/lo rows
  float* o;                // [B][d]
  float* hmlp;             // [B][F]
  float* rope_cs;          // [B][Dh/2][2]
  float* attn_part;        // [B][H] blocks of attn_pair_floats(nc_max, Dh)
  uint32_t* attn_count;    // [B][H]
  float* logits;           // [B][logits_ld]
  int32_t* tok;            // [B] token feeding the next depformer step
  float* y;                // [B][dd]
  float* yn;               // [B][max(dd, Fd)]
  float* dqkv;             // [B][3dd]
  float* dkv;              // [B][Ld][nq][2][dd]
  float* dout;             // [B][dd]
  float* dh;               // [B][Fd]
  // the depformer's batched user steps (steps 8..15, chunk c = step 8 + c)
  int32_t* tokb;           // [8][B] token feeding step 8 + c
  float* y_b;              // [8][B][dd]
  float* pz;               // [B][nq * dd] every step's in-projection of this tick's z
  float* dqkv_b;           // [8][B][3dd]
  float* dout_b;           // [8][B][dd]
  // bf16 hi/lo activation operands of the tensor-core contractions, [2*Bp][K]
  uint16_t* op_d;          // K = d   (normalised temporal stream)
  uint16_t* op_o;          // K = d   (attention output)
  uint16_t* op_f;          // K = F   (gated MLP hidden)
  uint16_t* op_z;          // K = d   (post final norm: text head and depformer input)
  uint16_t* op_dd;         // K = dd  (normalised depformer stream)
  uint16_t* op_do;         // K = dd  (depformer attention output)
  uint16_t* op_fd;         // K = Fd  (depformer gated hidden)
  uint16_t* op_ddb;        // [8][2*Bp][dd] the same three for the batched user steps
  uint16_t* op_dob;        // [8][2*Bp][dd]
  uint16_t* op_fdb;        // [8][2*Bp][Fd]
  float* ssq;              // fused-RMSNorm partial sums of squares [kMaxUnits][B]
  float* rstd_z;           // [B] 1/rms of the temporal output (text head and depformer input)
  // the persistent depformer: barrier words (count, generation, abort) and argmax partials
  unsigned long long* dkey;   // [2][B] fused-decision keys (text head, depformer heads)
  unsigned* dnan;          // [2]
  unsigned* dticket;       // [4]
  unsigned* pbar;          // [4]
  float* ppart_val;        // [kPMaxGrid][kPMaxB]
  int* ppart_idx;          // [kPMaxGrid][kPMaxB]
};

// The depformer step attention runs one warp per head in one CTA; its register use
// bounds the CTA to 512 threads (head dim 32 or 64) or 256 (head dim 128).
constexpr int kDepAttnMaxThreads(int head_dim) { return head_dim == 128 ? 256 : 512; }
constexpr int kDepAttnMaxHeads(int head_dim) { return kDepAttnMaxThreads(head_dim) / 32; }

// Engines of at most this many slots let each kernel's dependent launch right away
// (programmatic dependent launch) instead of after its main loop: at small B the next
// kernel's prologue and weight prefetch then overlap more of the tick (B=1 4.86 against
// 4.98 ms, B=8 7.09 against 7.15 ms), while at B=64 they compete with the running
// kernel (21.10 against 20.77 ms).
constexpr int kEarlyTriggerMaxB = 8;

constexpr int kMaxUnits = 4096;      // cap on (M-tile x K-split) units of one contraction
constexpr int kMaxSplits = 8;        // K-splits of one tile form one (portable) cluster
constexpr int kMaxTiles = 1024;      // cap on M-tiles of one contraction

// ---- programmatic dependent launch ------------------------------------------------------
// The tick's kernels are launched with programmatic stream serialization (unless
// PP_FLAG_NO_PDL): a kernel may start while its predecessor drains, and waits
// (griddepcontrol.wait) for the predecessor's completion and memory flush before it
// touches any data the predecessor may write.  The long kernels let their successor
// launch once their main work is done (pdl_trigger); the others trigger implicitly when
// they exit.  Without the launch attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_wait_and_trigger() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

extern bool g_use_pdl;          // set by the engine before it captures a tick
extern int g_launch_priority;    // nonzero: launch priority attribute of the next launches

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[3];
  int n = 0;
  if (g_launch_priority != 0) {
    at[n].id = cudaLaunchAttributePriority;
    at[n].val.priority = g_launch_priority;
    ++n;
  }
  if (g_use_pdl) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = (unsigned)cluster_x;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---- launchers (stream-ordered; return cudaGetLastError) ----------------------------
// op (may be null): also write the layer-0 operand hi/lo(alpha * x) and the sum of x^2
cudaError_t launch_begin(const Dims& D, const Buffers& b, const float* alpha, uint16_t* op,
                         float* ssq, cudaStream_t s);
// out (fp32, may be null) and/or op (bf16 hi/lo operand [2*Bp][K], may be null)
cudaError_t launch_rmsnorm(const Dims& D, const float* x, int ldx, const float* alpha, int K,
                           float* out, int ldo, uint16_t* op, cudaStream_t s);

// two values as packed bf16 (lo in the low half)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  // round to nearest even, NaN kept quiet
  uint32_t a = __float_as_uint(lo), b = __float_as_uint(hi);
  a = (a & 0x7FFFFFFFu) > 0x7F800000u ? 0x7FC00000u : a + 0x7FFFu + ((a >> 16) & 1u);
  b = (b & 0x7FFFFFFFu) > 0x7F800000u ? 0x7FC00000u : b + 0x7FFFu + ((b >> 16) & 1u);
  return (a >> 16) | (b & 0xFFFF0000u);
}

// hi = bf16(v) and lo = bf16(v - hi), both rounded to nearest even (NaN stays NaN)
__device__ __forceinline__ void bf16_split(float v, uint16_t& hi, uint16_t& lo) {
  uint32_t u = __float_as_uint(v);
  uint32_t h = (u & 0x7FFFFFFFu) > 0x7F800000u ? 0x7FC00000u : ((u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u);
  const float rem = v - __uint_as_float(h);
  uint32_t r = __float_as_uint(rem);
  r = (r & 0x7FFFFFFFu) > 0x7F800000u ? 0x7FC00000u : r + 0x7FFFu + ((r >> 16) & 1u);
  hi = (uint16_t)(h >> 16);
  lo = (uint16_t)(r >> 16);
}

// hi/lo split of v into operand row b (hi) and Bp + b (lo), column k
__device__ __forceinline__ void op_store(uint16_t* op, int ld, int Bp, int b, int k, float v) {
  uint16_t hi, lo;
  bf16_split(v, hi, lo);
  op[(size_t)b * ld + k] = hi;
  op[(size_t)(Bp + b) * ld + k] = lo;
}

// Greedy decision fused into a head contraction (the greedy-only tick): each CTA keeps,
// per slot, the best (value, lowest index) of the rows it finalises as one 64-bit key,
// and the last CTA to finish takes every slot's decision.
struct DecideArgs {
  int kind;                  // 0: none; 1: text row 0; 2: depformer row step + 1
  int step;                  // kind 2: the depformer step
  int V;                     // logits per row (the forced-token range is 0..V)
  int tokb;                  // kind 2: also write the batched steps' token table
  unsigned long long* key;   // [B] the launch's best key per slot, zero between launches
  unsigned* nan;             // [1] a NaN was seen
  unsigned* ticket;          // zero before the launch; left zero after it
  const int32_t* live;
  const uint8_t* fmask;
  const int32_t* forced;
  const int32_t* user;
  const int32_t* pos;
  int32_t* out_col;
  int32_t* tok;
  int32_t* tok_b;            // [8][B]
  int32_t* hist;             // kind 1: the repetition-penalty ring [B][hist_ld]
  int32_t* hist_len;
  int hist_ld;               // a power of two
};

// Tensor-core contraction (k_umma.cu).
struct RopeArgs {
  const int32_t* live;     // [B]
  const int32_t* pos;      // [B]
  const float* cs;         // [B][Dh/2][2] cos, sin of this tick's position
  float* q;                // [B][d] rotated query x log2(e)/sqrt(Dh)
  uint16_t* q_op;          // [B][H][2][Dh] the same as bf16 hi/lo rows
  uint16_t* ring;          // this layer's ring [B][2][H][W][Dh] bf16
  int d, H, Dh, W;
};

struct UmmaArgs {
  int halves;          // 128-row halves of the weight tile: 1 or 2 (a function of the shape)
  int early_trigger;   // let the next kernel launch at once (small engines), not after the main loop
  RopeArgs rope;       // EPI_ROPE
  int M;               // output rows (EPI_SILU: number of gate/up pairs)
  int pair_rows;       // EPI_SILU: F, the up rows start pair_rows after the gate rows; else 0
  int row0;            // first row of this matrix in the stacked weight tensor map
  int kblocks;         // ceil(K / 64)
  int splits;          // K-splits per M-tile (depends on shape and SM count only)
  int m_tiles;
  int B;               // slots
  int N;               // MMA N = 2 * Bp
  int epi;
  float* Y;            // EPI_STORE / EPI_ADD / EPI_EMB output [B][ldy]
  int ldy;
  const uint16_t* emb; // EPI_EMB table [rows][M]
  const int32_t* tok;
  uint16_t* op_out;    // EPI_SILU: operand [2*Bp_out][ld_op] of the next contraction
  int ld_op;
  int Bp_out;
  uint32_t* status;
  const int32_t* test_ctl;   // optional fault-test word (see pp_async.cuh)
  // Fused RMSNorm, producer side (EPI_ADD / EPI_EMB): besides y, write the next
  // contraction's operand hi/lo(norm_alpha * y) [2*Bp][M] and the sums of y^2 over each
  // row slice: ssq_out[(tile * splits + split) * B + b], one partial per CTA (the slice
  // of the tile's rows that CTA finalises; the whole tile when it is not split).
  const float* norm_alpha;
  uint16_t* norm_op;
  float* ssq_out;
  // Fused RMSNorm, consumer side: scale the contraction by 1/rms of the input, from the
  // producer's partials (ssq_in, ssq_nparts slices, width ssq_K) or precomputed
  // (rstd_in); block 0 also stores the values in rstd_out when it is given.
  const float* ssq_in;
  int ssq_nparts;
  int ssq_K;
  float eps;
  const float* rstd_in;
  float* rstd_out;
  // Independent column chunks (gridDim.y): chunk c runs the same contraction on its own
  // operand rows and writes its own outputs, each pointer advanced by c times its
  // stride below (0: the chunks share it).  Used for the depformer steps that run as
  // one batched pass.
  int chunks;
  int a_chunk_rows;        // weight rows between chunks (a different matrix per chunk)
  int b_chunk_rows;        // operand rows between chunks
  long long y_chunk;       // floats between chunks' Y
  long long op_chunk;      // elements between chunks' norm_op / op_out
  int ssq_out_chunk;       // floats between chunks' ssq_out
  int ssq_in_chunk;        // floats between chunks' ssq_in
  long long emb_chunk;     // elements between chunks' embedding tables
  int tok_chunk;           // entries between chunks' tokens
  DecideArgs dec;          // fused greedy decision (EPI_STORE heads; kind 0: none)
};
cudaError_t launch_umma(const UmmaArgs& a, const CUtensorMap& mA, const CUtensorMap& mB,
                        cudaStream_t s);
cudaError_t umma_setup(int N);

// EPI_ROPE (tensor-core path only): the temporal qkv contraction's rows are not stored;
// q and k are rotated at the slot's position (interleaved pairs), the scaled query goes
// to q / q_op and k, v are appended to the layer's ring as bf16, for open slots only.
enum GemvEpi { EPI_STORE = 0, EPI_ADD = 1, EPI_SILU = 2, EPI_EMB = 3, EPI_ROPE = 4 };
struct GemvArgs {
  const uint16_t* W;     // [M, K] bf16 (EPI_SILU: [2M, K], gate rows then up rows)
  int M, K;
  const float* X;        // [B, ldx] fp32
  int ldx;
  float* Y;              // [B, ldy] fp32
  int ldy;
  int epi;
  const uint16_t* emb;   // EPI_EMB: table [rows, M] bf16, row tok[b]
  const int32_t* tok;    // EPI_EMB
};
cudaError_t launch_gemv(const Dims& D, const GemvArgs& a, cudaStream_t s);

cudaError_t launch_rope_ring(const Dims& D, const Buffers& b, int layer, cudaStream_t s);
// Split-K ring attention (k_attn.cu): for slot s < B and head h < H,
//   out[s][h*Dh + i] = sum_j softmax_j(q_scale * q.K_j, base 2) V_j,  j < n_valid[s].
struct AttnArgs {
  const float* q;          // [B][q_ld], head h at h*Dh
  int q_ld;
  float q_scale;           // multiplies q; log2(e)/sqrt(Dh) for a plain softmax
  const uint16_t* k;       // head h of slot s: k + s*slot_stride + h*W*Dh, [W][Dh] bf16
  const uint16_t* v;
  size_t slot_stride;      // elements
  const int32_t* n_valid;  // [B]; values above W count as W, values <= 0 give zero output
  int H, W, nc_max;        // nc_max = ceil(W / kAttnChunk)
  float* out;              // [B][out_ld] fp32
  int out_ld;
  uint16_t* op;            // optional bf16 hi/lo operand [2*op_Bp][H*Dh]
  int op_Bp;
  float* part;             // scratch [B*H] blocks of attn_pair_floats(nc_max, Dh)
  uint32_t* count;         // scratch [B*H], zero before the call; left zero after it
  uint32_t* status;        // optional: PP_S_TIMEOUT is raised here when a wait gives up
  const int32_t* test_ctl; // optional fault-test word (see pp_async.cuh)
  int early_trigger;       // tensor-core kernel: let the next kernel launch at once (small
                           // engines), not at the end
  uint16_t* q_op;          // head dim 128: bf16 hi/lo query operand [B*H*2][Dh], already
                           // scaled by q_scale (the tensor-core kernel reads only this)
};
// Tensor maps of the tensor-core attention (head dim 128): K and V as 4-D [slot][H][W][Dh]
// bf16 (box 64 x 128 rows), the query operand as 2-D [B*H*2][Dh] (box 64 x 2 rows),
// all with the 128-byte swizzle.
struct AttnMaps {
  CUtensorMap k, v, q;
};
bool attn_maps(AttnMaps* m, const uint16_t* k, const uint16_t* v, size_t slot_stride, int slots,
               int H, int W, int Dh, const uint16_t* q_op, int pairs);
// Head dim 128 runs on the tensor cores (maps and a.q_op required; slot_base is the slot
// coordinate of slot 0 in the K/V maps); head dims 32 and 64 run on the CUDA cores.
cudaError_t launch_attn_args(const AttnArgs& a, int B, int Dh, const AttnMaps* maps,
                             int slot_base, cudaStream_t s);
cudaError_t launch_attn_cc(const AttnArgs& a, int B, int Dh, cudaStream_t s);
cudaError_t launch_attn_tc(const AttnArgs& a, int B, const AttnMaps& maps, int slot_base,
                           cudaStream_t s);
// q_op[(s*H + h)*2 + {0,1}][i] = hi/lo of q_scale * q[s][h*Dh + i]
cudaError_t launch_q_split(const AttnArgs& a, int B, int Dh, cudaStream_t s);
cudaError_t launch_attn(const Dims& D, const Buffers& b, int layer, bool op, const AttnMaps* maps,
                        cudaStream_t s);
cudaError_t launch_text_argmax(const Dims& D, const Buffers& b, cudaStream_t s);
cudaError_t launch_dep_attn(const Dims& D, const Buffers& b, int step, int layer, bool op,
                            cudaStream_t s);
cudaError_t launch_dep_argmax(const Dims& D, const Buffers& b, int step, cudaStream_t s);
// The depformer as one persistent kernel (k_dep_persist.cu, PP_FLAG_LOW_LATENCY).
constexpr int kPMaxB = 8;        // slots of an engine that runs it
constexpr int kPMaxGrid = 256;   // CTAs (one per SM)
struct PersistArgs {
  Dims D;
  Buffers b;
  unsigned* bar_count;   // grid barrier: arrivals and generation, zeroed before each launch
  unsigned* bar_gen;
  int* abort;            // set by a CTA whose barrier wait gave up
  float* part_val;       // [kPMaxGrid][kPMaxB] per-CTA argmax partials of a head
  int* part_idx;         // index | 0x80000000 when the CTA saw a NaN
};
size_t persist_smem(const Dims& D);
cudaError_t persist_setup(const Dims& D);
cudaError_t launch_dep_persist(const PersistArgs& p, cudaStream_t s);

// attention of the batched user steps of one depformer layer
cudaError_t launch_dep_attn_batch(const Dims& D, const Buffers& b, int layer, cudaStream_t s);
// Depformer input of `chunks` consecutive steps from k0 (b.pz + the token tables): y, the
// first layer's operand and one sum of y^2 per slot and step (b.ssq[c * B + s]).
cudaError_t launch_dep_in(const Dims& D, const Buffers& b, int k0, int chunks, const int32_t* tok,
                          const uint16_t* emb, long long emb_chunk, float* y, long long y_chunk,
                          uint16_t* op, long long op_chunk, cudaStream_t s);
constexpr int kDepBatch = 8;   // user steps run as one batched pass (n_q / 2)
cudaError_t sample_setup(const Dims& D);   // shared-memory opt-in of the decision kernels
cudaError_t launch_sample_rows(const float* logits, int64_t ld, int rows, int n, float temperature,
                               int top_k, float top_p, float penalty, const int32_t* hist,
                               int hist_ld, const int32_t* hist_n, const float* uniforms,
                               int32_t* tokens, uint32_t* status, cudaStream_t s);
cudaError_t launch_finish(const Dims& D, const Buffers& b, cudaStream_t s);
cudaError_t launch_user_rows(const Dims& D, const Buffers& b, cudaStream_t s);

}  // namespace pp
