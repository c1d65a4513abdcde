/*
 * pp.h - C ABI of the GB300 (sm_103a) lockstep decode tick of the PersonaPlex / Moshi
 * RQ-Transformer: one 80 ms step for up to max_batch concurrent full-duplex sessions.
 *
 * What one step computes (vllm-omni recipes/NVIDIA/PersonaPlex.md, "Architecture";
 * "PersonaPlex 全双工语音对话实战 ... 80ms Lockstep", sections 架构 and 帧 token 布局):
 *   1. x = text_table[col[0]] + sum_{r=1..16} audio_table[r-1][col[r]] over the
 *      previous column (row 0 inner-monologue text, rows 1-8 agent audio, rows 9-16
 *      user audio);
 *   2. the Helium temporal transformer (fp32-alpha RMSNorm, fused QKV in-projection,
 *      interleaved RoPE at the slot's absolute position, attention over the slot's
 *      ring KV cache with a sliding window, SiLU-gated MLP);
 *   3. the greedy text token (lowest index on ties) unless forced;
 *   4. the depformer: 16 autoregressive codebook steps with a cache reset every frame;
 *      agent rows 1-8 greedy unless forced, user rows 9-16 always the incoming codes.
 * Persona and voice prefill are ordinary steps with forced tokens.
 *
 * Conventions
 *  - Every array is indexed by slot: [max_batch, ...], row-major.  Slots that are not
 *    open are ignored on input and produce column rows of -1 on output.
 *  - Weights and workspace are caller-owned device memory; the engine never frees
 *    them and they must outlive the engine.  Matrices are row-major [out, in] bf16
 *    (PyTorch Linear orientation); per-layer tensors are stacked along a leading axis.
 *  - Return value: PP_OK (0) or a negative PP_E* code, detected synchronously on the
 *    host.  Conditions found on the device (NaN logits, out-of-range tokens, timed-out
 *    waits) are OR-ed into a device status word read by pp_status.
 *  - A stream argument is a cudaStream_t passed as void* (NULL = legacy default stream).
 */
#ifndef PP_H
#define PP_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PP_ROWS 17           /* rows of one column: text, 8 agent codebooks, 8 user codebooks */
#define PP_AGENT_ROWS 8
#define PP_USER_ROWS 8

/* host-detected errors */
#define PP_OK 0
#define PP_EINVAL (-1)       /* bad argument or config */
#define PP_E_BUSY (-2)       /* slot already open */
#define PP_E_RANGE (-3)      /* slot, layer or position out of range */
#define PP_E_NOTLIVE (-4)    /* slot not open */
#define PP_E_CUDA (-5)       /* a CUDA runtime call failed */
#define PP_E_NOSPACE (-6)    /* workspace smaller than pp_workspace_bytes */

/* device-detected conditions (bits of the status word) */
#define PP_S_NAN 0x1u        /* a logit row held NaN (the NaN entries were not chosen) */
#define PP_S_INDEX 0x2u      /* an input token was out of range (replaced by the initial token) */
#define PP_S_TIMEOUT 0x4u    /* a bounded device-side wait gave up: that tick's columns
                                and logits are undefined, and so are the ring entries it
                                wrote, so the sessions open during it should be closed and
                                reopened; the next tick itself starts clean */

typedef struct {
  int32_t d_model;       /* 4096 */
  int32_t n_layers;      /* 32 */
  int32_t n_heads;       /* 32; head dim = d_model / n_heads, one of 32, 64, 128 */
  int32_t ffn;           /* 11008 */
  int32_t text_vocab;    /* 32000 text logits; text tables have text_vocab+1 rows, the
                            last being TEXT_INITIAL_TOKEN = text_vocab */
  int32_t audio_card;    /* 2048 codes; audio tables have audio_card+1 rows, the last
                            being AUDIO_INITIAL_TOKEN = audio_card */
  int32_t n_q;           /* 16 audio rows = depformer steps (must be 16) */
  int32_t dep_d;         /* 1024 */
  int32_t dep_layers;    /* 6 */
  int32_t dep_heads;     /* 16; head dim = dep_d / dep_heads, one of 32, 64, 128; at most
                            16 heads (8 with head dim 128) */
  int32_t dep_ffn;       /* depformer FFN width */
  int32_t window;        /* 3000 ring positions per slot */
  int32_t max_batch;     /* slots, 1..64 */
  float eps;             /* RMSNorm epsilon (inside the square root) */
  float rope_base;       /* RoPE base (10000) */
  int32_t flags;         /* PP_FLAG_* bits; 0 = default */
} pp_config;

/* Weight contractions on CUDA cores (fp32 activations) instead of the default
 * tcgen05 tensor-core path (split-bf16 activations).  The two paths round
 * differently, so a session's bits are reproducible within one path only. */
#define PP_FLAG_CUDA_CORE_GEMM 0x1
/* Launch the tick's kernels without programmatic dependent launch.  By default each
 * kernel may start while its predecessor drains: a contraction allocates its tensor
 * memory and streams its first weight tiles (weights never depend on the previous
 * kernel), then waits for the predecessor before it reads any activation.  In engines
 * of at most 8 slots a contraction or attention kernel releases its successor as soon as
 * it starts, in larger ones after its main loop. */
#define PP_FLAG_NO_PDL 0x2
/* Split an engine of 16 or more slots into two groups that run as parallel branches of
 * the tick graph, so one group's latency-bound depformer can overlap the other's
 * bandwidth-bound attention (weights are then streamed once per group).  Off by
 * default: on GB300 the doubled weight traffic cost more than the overlap saved.
 * Grouping never changes a session's bits. */
#define PP_FLAG_TWO_GROUPS 0x4
/* Run depformer steps 0..7 only.  Steps 8..15 decide user rows 9..16, which always take
 * the incoming user codes, so every column is unchanged; only their logits (the last 8
 * codebook blocks of the logits output) are not computed and keep stale values.  Off by
 * default: the default tick runs all 16 steps. */
#define PP_FLAG_SKIP_USER_STEPS 0x8
/* Run depformer steps 8..15 one at a time, as steps 0..7 are.  By default (tensor-core
 * path) they run as one batched pass: once step 7 has decided row 8, the tokens of steps
 * 8..15 are known (row 8, then the user codes of rows 9..15), so each contraction and the
 * step attention process the 8 steps together while every step computes exactly what it
 * computes alone (its own in-projection and head, causal attention over steps 0..k of
 * the frame).  Columns and logits agree with the one-at-a-time schedule to fp32
 * rounding (the batched contractions may split K differently). */
#define PP_FLAG_SEQUENTIAL_USER_STEPS 0x10
/* Weight tiles of 256 rows for the temporal layers' matrices and the text head: two
 * 128-row halves share each activation tile, one CTA (one copy producer) per SM.  Off by
 * default: on GB300 it measured slower (B=64 tick 22.57 ms against 21.24 ms with the
 * default 128-row tiles, two CTAs per SM), since a producer streams only about 30 GB/s
 * and two producers per SM stream twice that.  The tile height changes the K-split, so
 * a session's bits are reproducible within one setting only. */
#define PP_FLAG_WIDE_TILES 0x20
/* Low-latency depformer for small engines (max_batch <= 8, tensor-core path): the 16
 * codebook steps run as one persistent kernel, one CTA per SM, phases separated by a
 * bounded grid barrier, contractions on the CUDA cores in fp32.  It replaces ~300
 * dependent launches per tick.  Its rounding differs from the default path, so a
 * session's bits are reproducible among engines with this flag.  Audio sampling is not
 * available with it (pp_session_sampling returns PP_EINVAL for audio_temperature > 0).
 * pp_create returns PP_EINVAL for max_batch > 8 or with PP_FLAG_CUDA_CORE_GEMM. */
#define PP_FLAG_LOW_LATENCY 0x40

/* Weight tensors (device pointers).  Shapes use d = d_model, L = n_layers, F = ffn,
 * Vt = text_vocab, Va = audio_card, dd = dep_d, Ld = dep_layers, Fd = dep_ffn. */
enum pp_weight {
  PP_W_EMB_TEXT = 0,     /* bf16 [Vt+1, d] */
  PP_W_EMB_AUDIO,        /* bf16 [n_q, Va+1, d]       (row r of a column uses table r-1) */
  PP_W_ATTN_ALPHA,       /* f32  [L, d] */
  PP_W_QKV,              /* bf16 [L, 3d, d]           rows: q heads, k heads, v heads */
  PP_W_O,                /* bf16 [L, d, d] */
  PP_W_MLP_ALPHA,        /* f32  [L, d] */
  PP_W_GU,               /* bf16 [L, 2F, d]           rows: gate (F) then up (F) */
  PP_W_DOWN,             /* bf16 [L, d, F] */
  PP_W_OUT_ALPHA,        /* f32  [d] */
  PP_W_TEXT,             /* bf16 [Vt, d] */
  PP_W_DEP_INPROJ,       /* bf16 [n_q, dd, d]         per-codebook input projection */
  PP_W_DEP_EMB_TEXT,     /* bf16 [Vt+1, dd]           step 0 token table */
  PP_W_DEP_EMB_AUDIO,    /* bf16 [n_q-1, Va+1, dd]    step k >= 1 uses table k-1 */
  PP_W_DEP_ATTN_ALPHA,   /* f32  [Ld, dd] */
  PP_W_DEP_QKV,          /* bf16 [Ld, 3dd, dd] */
  PP_W_DEP_O,            /* bf16 [Ld, dd, dd] */
  PP_W_DEP_MLP_ALPHA,    /* f32  [Ld, dd] */
  PP_W_DEP_GU,           /* bf16 [Ld, 2Fd, dd] */
  PP_W_DEP_DOWN,         /* bf16 [Ld, dd, Fd] */
  PP_W_DEP_OUT_ALPHA,    /* f32  [dd] */
  PP_W_DEP_HEADS,        /* bf16 [n_q, Va, dd]        per-codebook output head */
  PP_W_COUNT
};

typedef struct {
  const void* ptr[PP_W_COUNT];  /* device pointers, 16-byte aligned */
} pp_weights;

typedef struct pp_engine pp_engine;  /* opaque */

/* Shape of weight tensor `which` for config c: dims[0..*ndim-1], *is_f32 = 1 for the
 * fp32 alpha vectors, 0 for bf16.  Returns PP_EINVAL for a bad config or index. */
int pp_weight_shape(const pp_config* c, int which, int64_t dims[4], int* ndim, int* is_f32);

/* Bytes of device workspace the engine needs for config c (ring KV for every slot,
 * activations, per-step scratch, status word), or 0 for a bad config. */
size_t pp_workspace_bytes(const pp_config* c);

/* Create an engine: the RQ-Transformer of the config (vllm-omni
 * recipes/NVIDIA/PersonaPlex.md, "Architecture": Helium temporal transformer, depformer
 * over the 16 codebooks, the [B, 17, 1] column per 80 ms frame) serving up to max_batch
 * sessions in lockstep (same page, "Notes": elastic batching over a fixed set of slots;
 * mhpq 运维要点, one ring KV per slot).
 * w: device weight pointers (not copied, must outlive the engine).
 * workspace: device memory of at least pp_workspace_bytes(c) bytes, 256-byte aligned,
 * owned by the caller.  Captures the whole tick as one CUDA graph.  All slots start
 * closed.  Errors: PP_EINVAL, PP_E_NOSPACE, PP_E_CUDA. */
int pp_create(const pp_config* c, const pp_weights* w, void* workspace, size_t ws_bytes,
              pp_engine** out);

/* Release the engine's host state, its CUDA graph, streams and events.  The weights and
 * the workspace stay the caller's (they are not freed).  Work still queued on the
 * caller's streams must have finished.  NULL is ignored.  No counterpart on the pages
 * beyond the engine's lifetime. */
void pp_destroy(pp_engine* e);

/* Open slot `slot` for a new session at position 0: admission of a session into the
 * lockstep batch (vllm-omni PersonaPlex recipe, "Notes": sessions join and leave an
 * elastic batch, and a recycled slot is bit-exact with a fresh engine; mhpq 运维要点,
 * per-slot recycle).  The slot's ring contents are ignored from then on because
 * attention reads only positions written since open, so a recycled slot behaves exactly
 * like a fresh engine.  Takes effect at the next pp_step.
 * Errors: PP_E_RANGE (slot >= max_batch), PP_E_BUSY (already open). */
int pp_session_open(pp_engine* e, int slot);

/* Close slot `slot` at the next pp_step: the session leaves the elastic batch (same
 * passages as pp_session_open); from then on the slot's column rows are -1 and it
 * writes no KV.  Errors: PP_E_RANGE, PP_E_NOTLIVE. */
int pp_session_close(pp_engine* e, int slot);

/* Open slot `slot` resuming a session at absolute position pos (0 <= pos < 2^31-1):
 * the caller has already written the session's ring contents through pp_ring_block
 * (ring index j holds the latest position p < pos with p mod window = j).
 * Errors: PP_E_RANGE, PP_E_BUSY. */
int pp_session_import(pp_engine* e, int slot, int64_t pos);

/* Current absolute position of an open slot (frames since open), from the host
 * mirror.  Errors: PP_E_RANGE, PP_E_NOTLIVE. */
int pp_session_pos(pp_engine* e, int slot, int64_t* pos);

/* ---- sampling variants -------------------------------------------------------------
 * The pages decode greedily ("PersonaPlex ... vLLM-Omni", greedy decoding and parity:
 * the parity gates pin greedy output) and list the knobs a deployment may turn instead:
 * temperature, nucleus top-p and a repetition penalty for the text stream, a separate
 * audio temperature (deployment config; the persona-tuning article's generation
 * parameters).  A row that is sampled takes these steps in order:
 *   1. repetition penalty (text only): each distinct token among the session's last
 *      penalty_window text tokens has its logit divided by R when positive and
 *      multiplied by R otherwise (Keskar et al., CTRL, 2019);
 *   2. division by the temperature;
 *   3. top-k: keep the values at or above the k-th largest (ties kept);
 *   4. e_i = exp(v_i - max v) over the kept values;
 *   5. nucleus: keep e at or above the largest e value whose own mass plus the mass of
 *      every larger e reaches top_p * sum(e) (ties kept);
 *   6. inverse CDF in index order: the first kept token whose running mass exceeds
 *      u * (kept mass).
 * u is drawn from Philox4x64-10 (Salmon et al., SC 2011) under the key (seed, 0) at the
 * counter (position, row / 4, 0, 0): the top 24 bits of word row % 4, times 2^-24,
 * where row is 0 for text and 1..8 for the agent audio codebooks and position is the
 * session's position of the tick.  A session's draws thus depend on its seed and
 * position only, never on its slot.  Forced rows draw nothing.  Logits that are not
 * finite are never chosen.  Every decision is deterministic (fixed reduction orders). */
typedef struct {
  float text_temperature;    /* <= 0: the text row stays greedy (the default) */
  int32_t text_top_k;        /* <= 0: no top-k filter */
  float text_top_p;          /* in (0, 1]; 1: no nucleus filter */
  float repetition_penalty;  /* > 0; 1: off */
  int32_t penalty_window;    /* last N text tokens of the session, 0..256 */
  float audio_temperature;   /* <= 0: the agent audio rows stay greedy (the default) */
  int32_t audio_top_k;       /* <= 0: no top-k filter */
  float audio_top_p;         /* in (0, 1]; 1: no nucleus filter */
  uint64_t seed;             /* the session's random stream */
} pp_sampling;

/* Set the sampling parameters of open slot `slot` from its next tick on (NULL: greedy,
 * which is also the state after pp_session_open).  The text history behind the
 * penalty counts every text token of the session since open, forced ones included.
 * Errors: PP_E_RANGE, PP_E_NOTLIVE, PP_EINVAL (a NaN or out-of-range field, or text
 * sampling on a vocabulary above 51200 / audio sampling on a codebook above 51200). */
int pp_session_sampling(pp_engine* e, int slot, const pp_sampling* p);

/* Sample one token per row of device logits with caller-given uniforms, by the steps
 * above (the kernel the tick runs for a sampled row), asynchronous on `stream`:
 *   logits    f32 [rows, ld], row r's n logits at r*ld (n <= ld, n <= 51200)
 *   hist      int32 [rows, hist_ld] history tokens (order irrelevant) or NULL;
 *             hist_n int32 [rows] how many of row r's entries count (<= hist_ld <= 256)
 *   uniforms  f32 [rows] in [0, 1)
 *   tokens    int32 [rows] out
 *   status    optional device word; PP_S_NAN is OR-ed in when a row held NaN
 * temperature > 0, top_p in (0, 1], penalty > 0.  rows == 0 does nothing.
 * Errors: PP_EINVAL, PP_E_CUDA. */
int pp_sample(const float* logits, int64_t ld, int rows, int n, float temperature, int top_k,
              float top_p, float penalty, const int32_t* hist, int hist_ld,
              const int32_t* hist_n, const float* uniforms, int32_t* tokens, uint32_t* status,
              void* stream);

/* Device address of one ring block: layer `layer`, slot `slot`, kv = 0 (K, stored
 * after RoPE) or 1 (V); the block is bf16 [n_heads, window, head_dim], contiguous.
 * Errors: PP_E_RANGE, PP_EINVAL. */
int pp_ring_block(pp_engine* e, int layer, int slot, int kv, void** ptr);

/* One lockstep tick for every open slot, asynchronous on `stream`.  Device pointers:
 *   prev_column   int32 [max_batch, 17]  the previous column (for a fresh session:
 *                                         [text_vocab, audio_card x 16])
 *   user_codes    int32 [max_batch, 8]   this frame's user codes -> rows 9..16
 *   force_mask    uint8 [max_batch, 17]  nonzero: rows 0..8 take forced_tokens
 *                                         (rows 9..16 ignore it); may be NULL
 *   forced_tokens int32 [max_batch, 17]  may be NULL when force_mask is NULL
 *   column        int32 [max_batch, 17]  out: this frame's column (-1 for closed slots)
 *   logits        f32 [max_batch, text_vocab + n_q*audio_card] out, or NULL: text
 *                 logits then the 16 depformer steps' logits
 * Open slots advance one position.  Errors: PP_EINVAL, PP_E_CUDA. */
int pp_step(pp_engine* e, const int32_t* prev_column, const int32_t* user_codes,
            const uint8_t* force_mask, const int32_t* forced_tokens, int32_t* column,
            float* logits, void* stream);

/* The same tick with HOST buffers (same layouts; pinned memory recommended): copies
 * the inputs to the device, runs the tick and copies the column (and logits if not
 * NULL) back, on `stream`, returning after the results are on the host. */
int pp_step_host(pp_engine* e, const int32_t* prev_column, const int32_t* user_codes,
                 const uint8_t* force_mask, const int32_t* forced_tokens, int32_t* column,
                 float* logits, void* stream);

/* Wait for `stream`, then read and clear the device status word into *bits
 * (PP_S_* flags).  The pages define no error reporting; the conditions are this
 * library's (an index or NaN the greedy decision of the recipe's "Notes" would meet, a
 * bounded wait).  Deliberately an out-parameter rather than a return value, so that the
 * return value stays the host-side error code of every other call.
 * Errors: PP_E_CUDA. */
int pp_status(pp_engine* e, void* stream, uint32_t* bits);

/* Number of kernel launches one greedy pp_step makes (the nodes of the captured greedy
 * graph).  The engine holds two graphs of the tick: while no open slot samples, pp_step
 * runs the greedy one, whose text and depformer heads take their decisions in their own
 * epilogues (the last CTA of each head reduces every CTA's best (value, lowest index)
 * key); with a sampled slot open it runs the one with the decision kernels.  Both give a
 * greedy slot the same bits. */
int pp_step_kernel_count(pp_engine* e);

/* ---- failure-detection tests --------------------------------------------------------
 * Lets a test make the tick's bounded device-side waits run out without faulting the
 * GPU: it lowers the poll budget of every bounded wait and asks producers of the named
 * kernel families to withhold copies, so that a consumer's wait on a copy that never
 * comes gives up, the kernel raises PP_S_TIMEOUT, drains its copies, frees its tensor
 * memory and returns.  This call has no counterpart on the pages.
 *   wait_polls  poll budget of each bounded wait; 0 restores the default (2^24 polls,
 *               seconds); a wait reads it only after 1024 unsuccessful polls
 *   withhold    copies still to withhold: the first producer of a named family to start
 *               takes one (its first activation tile in a contraction, its first V tile
 *               in the attention), and so on until none are left; 0 withholds nothing
 *   kinds       PP_TEST_UMMA, PP_TEST_ATTN and/or PP_TEST_PERSIST
 * Stream-ordered on `stream`; the engine's graph is unchanged.  Reset with (0, 0, 0)
 * after the test.  Errors: PP_EINVAL, PP_E_CUDA. */
#define PP_TEST_UMMA 0x1   /* the tensor-core weight contractions */
#define PP_TEST_ATTN 0x2   /* the ring attention (both kernels) */
#define PP_TEST_PERSIST 0x4 /* the persistent depformer: a CTA leaves before its first
                               grid barrier, so the others' barrier waits run out */
int pp_test_faults(pp_engine* e, int32_t wait_polls, int32_t withhold, int32_t kinds,
                   void* stream);

/* Kernel families of one tick, for pp_profile_step. */
enum pp_kernel_kind {
  PP_K_BEGIN = 0,   /* control + 17-table embedding sum + RoPE angle table */
  PP_K_NORM,        /* RMSNorm of the temporal stream */
  PP_K_QKV,         /* fused QKV in-projection (tensor-core path: with RoPE + ring-KV write) */
  PP_K_ROPE_RING,   /* RoPE + ring-KV write (CUDA-core path) */
  PP_K_ATTN,        /* split-K sliding-window ring attention (+ chunk merge) */
  PP_K_OPROJ,       /* out-projection + residual */
  PP_K_GATEUP,      /* gate/up projection + SiLU gating */
  PP_K_DOWN,        /* down-projection + residual */
  PP_K_TEXT_HEAD,   /* final norm, text head, greedy text token */
  PP_K_DEP_INPROJ,  /* depformer: input projections (tensor-core path: all codebooks in one
                       launch, then each step's token embedding) */
  PP_K_DEP_NORM,    /* depformer: RMSNorms */
  PP_K_DEP_QKV,     /* depformer: QKV projection */
  PP_K_DEP_ATTN,    /* depformer: attention over the frame's steps */
  PP_K_DEP_OPROJ,   /* depformer: out-projection + residual */
  PP_K_DEP_GATEUP,  /* depformer: gate/up projection + SiLU gating */
  PP_K_DEP_DOWN,    /* depformer: down-projection + residual */
  PP_K_DEP_HEAD,    /* depformer: per-codebook head + greedy / forced / user row */
  PP_K_FINISH,      /* end-of-tick bookkeeping */
  PP_K_DEP_PERSIST, /* depformer: all 16 steps in one persistent kernel (PP_FLAG_LOW_LATENCY) */
  PP_K_COUNT
};

/* pp_step (same arguments) through a second captured graph that records a timing
 * event at every kernel boundary; waits for the tick, then ADDS each kernel's
 * duration (ms, event to event, so it includes the launch gap before the next
 * kernel) to kind_ms[kind] and its launch count to kind_launches[kind] (both arrays of
 * PP_K_COUNT entries, caller-owned host memory).  For measurement only: slower than
 * pp_step.  Errors: PP_EINVAL, PP_E_CUDA. */
int pp_profile_step(pp_engine* e, const int32_t* prev_column, const int32_t* user_codes,
                    const uint8_t* force_mask, const int32_t* forced_tokens, int32_t* column,
                    float* logits, void* stream, double* kind_ms, int64_t* kind_launches);

/* ---- the tick's attention as a standalone call ---------------------------------------
 * Split-K sliding-window decode attention over ring blocks, the kernel each layer of
 * pp_step runs (vllm-omni recipe, "Architecture": a 3000-frame sliding window held in a
 * ring KV cache per slot).  For slot s < B and head h < H:
 *   out[s][h*D + i] = sum_{j < n_valid[s]} softmax_j(q[s][h] . K_j / sqrt(D)) V_j[i]
 * over ring indices j (softmax does not depend on key order, so the ring need not be
 * rotated); n_valid[s] == 0 gives zeros.  Reductions run in a fixed order set by the
 * ring index alone, so every slot's result is independent of the others.  D = 128 runs
 * on the tensor cores: q / sqrt(D) and the softmax weights enter them as bf16 hi/lo
 * pairs (about 16 significant bits; relative error ~1e-5 against fp64); D = 32 and 64
 * run on the CUDA cores in fp32.
 *   q          f32 [B][H][D], device, 16-byte aligned
 *   k, v       bf16: head h of slot s is the [W][D] block at k + s*slot_stride + h*W*D
 *              (elements), device, 16-byte aligned, slot_stride a multiple of 8; for
 *              D = 128 the blocks are read through a tensor map, and a layout the map
 *              cannot describe returns PP_EINVAL
 *   n_valid    int32 [B], device; values above W count as W, values <= 0 give zeros
 *   out        f32 [B][H*D], device
 *   status     optional device word (may be NULL): PP_S_TIMEOUT is OR-ed into it when a
 *              bounded wait inside the kernel gave up (the output is then incomplete);
 *              with NULL such a timeout goes unreported
 *   scratch    device memory of at least pp_ring_attention_scratch_bytes(B, H, D, W)
 *              bytes, 256-byte aligned, caller-owned; its contents need no set-up
 * D (head_dim) is 32, 64 or 128.  Asynchronous on `stream`.  Errors: PP_EINVAL,
 * PP_E_NOSPACE (scratch too small), PP_E_CUDA. */
size_t pp_ring_attention_scratch_bytes(int B, int H, int head_dim, int window);
int pp_ring_attention(const float* q, const uint16_t* k, const uint16_t* v, int64_t slot_stride,
                      const int32_t* n_valid, int B, int H, int head_dim, int window,
                      float* out, uint32_t* status, void* scratch, size_t scratch_bytes,
                      void* stream);

/* pp_ring_attention for callers that cannot allocate device memory or pass scratch:
 * for example a host whose device memory all belongs to a pooling allocator that a
 * library must not bypass or grow, or a real-time frame loop in which an allocation
 * (it can synchronise the device and take milliseconds) would break the 80 ms cadence.
 * The pages have no counterpart to this call; it exists for those callers.
 * Same arguments and result as pp_ring_attention, minus the scratch: the partials and
 * tickets live in one device array built into the library (27,795,456 bytes, about
 * 26.5 MiB, held on every GPU that loads the library until the process exits).  Limits: B*H <= 2048,
 * window <= 3072, head_dim <= 128; larger sizes return PP_E_RANGE.  The first call on
 * a device looks up the array's device address (make that first call before any
 * stream capture).  Every call shares the array, so calls that overlap on the GPU
 * (other streams, other threads) race; each call resets the tickets it needs.
 * Allocates no memory.  Errors: PP_EINVAL, PP_E_RANGE, PP_E_CUDA. */
int pp_ring_attention_noalloc(const float* q, const uint16_t* k, const uint16_t* v,
                              int64_t slot_stride, const int32_t* n_valid, int B, int H,
                              int head_dim, int window, float* out, uint32_t* status,
                              void* stream);

/* ---- session driver: host bookkeeping around pp_step ------------------------------
 * Admission and recycle of slots, the persona / voice prefill and the acoustic delay,
 * all on the host (no device memory).  Sessions exchange ALIGNED frames with the
 * driver: one frame = the 8 codes of one 80 ms Mimi frame (and, for the agent, its text
 * token).  In the model's columns the acoustic codebooks 1..7 of each stream run one
 * frame behind codebook 0 and the text (mhpq 3.3, "80 ms frame + 80 ms acoustic
 * delay"), so the driver feeds the user rows of tick t as [U_t[0], U_{t-1}[1..7]] and
 * returns agent frame f = (text and codebook 0 of tick f, codebooks 1..7 of tick f+1),
 * one tick late.  The initial token (audio_card) stands in for frame -1.
 * Prefill (mhpq, "Persona Voice 注入": voice + 2 x silence + persona): n_voice ticks of
 * voice-prompt frames, silence_ticks of silence, n_persona ticks with the text row
 * forced to the persona tokens (audio silent), silence_ticks of silence, then live.
 * Forced agent frames are shifted exactly like generated ones. */
typedef struct pp_driver pp_driver;

typedef struct {
  const int32_t* voice_frames;    /* [n_voice][8] aligned voice-prompt codes, host (copied) */
  int n_voice;
  const int32_t* persona_tokens;  /* [n_persona] text tokens, host (copied) */
  int n_persona;
  const int32_t* silence_frame;   /* [8] aligned codes of one silence frame, host (copied);
                                     NULL: the initial token in every codebook */
  int silence_ticks;              /* length of each of the two silence stretches */
} pp_prompt;

enum { PP_DRV_FREE = 0, PP_DRV_VOICE = 1, PP_DRV_SILENCE = 2, PP_DRV_PERSONA = 3,
       PP_DRV_LIVE = 4 };

/* A driver for an engine of max_batch slots.  Errors: PP_EINVAL. */
int pp_driver_create(int max_batch, int text_vocab, int audio_card, pp_driver** out);
void pp_driver_destroy(pp_driver* d);

/* Admit a session into the lowest free slot (*slot), also opening it on `e` when e is
 * not NULL.  Codes must lie in [0, audio_card], text tokens in [0, text_vocab].
 * Errors: PP_EINVAL, PP_E_BUSY (no free slot), or pp_session_open's error. */
int pp_driver_open(pp_driver* d, pp_engine* e, const pp_prompt* prompt, int* slot);

/* End the session in `slot` (and close it on `e` when not NULL); the slot is free for
 * the next admission.  Errors: PP_EINVAL, PP_E_RANGE, PP_E_NOTLIVE. */
int pp_driver_close(pp_driver* d, pp_engine* e, int slot);

/* Phase of the slot's next tick (PP_DRV_*), or PP_EINVAL / PP_E_RANGE. */
int pp_driver_phase(const pp_driver* d, int slot);

/* Inputs of the next pp_step from this tick's aligned user frames [max_batch][8]: all
 * host buffers of pp_step's layouts.  Does not change the driver.  Errors: PP_EINVAL
 * (NULL buffer, or a user code outside [0, audio_card] in an open slot). */
int pp_driver_prepare(pp_driver* d, const int32_t* user_frames, int32_t* prev_column,
                      int32_t* user_codes, uint8_t* force_mask, int32_t* forced);

/* Take the tick's output column [max_batch][17] (host) and the same user frames;
 * writes agent_frames [max_batch][9] (text + 8 codes): the frame this tick completed,
 * or -1 in every entry when none (a closed slot, or a session's first tick).  Advances
 * every open slot by one tick.  Errors: PP_EINVAL. */
int pp_driver_absorb(pp_driver* d, const int32_t* user_frames, const int32_t* column,
                     int32_t* agent_frames);

/* prepare + pp_step_host + absorb on engine `e`; column_out [max_batch][17] may be
 * NULL.  Blocks until the tick's results are on the host.  Errors: as the three. */
int pp_driver_tick(pp_driver* d, pp_engine* e, const int32_t* user_frames,
                   int32_t* agent_frames, int32_t* column_out, void* stream);

/* ---- Mimi RVQ dequantisation: codes to latent, the first step after the tick ---------
 * The agent's audio rows of each output column are Mimi codes: residual vector
 * quantisation with 8 codebooks of 2048 entries at 12.5 Hz (mhpq, section 2.3 "Mimi";
 * Recipe, Architecture).  The codec decoder starts from their latent, which is the sum
 * of the selected entries:
 *   out[f][d] = sum_{k < n_books} codebooks[k][codes[f*code_stride + k]][d]
 * added in codebook order in fp32.
 *   codes      int32, device, 4-byte aligned; frame f's codes at codes + f*code_stride.
 *              For a pp_step output column [B][17], pass codes = column + 1 and
 *              code_stride = 17: the agent rows 1..8.
 *   codebooks  f32 [n_books][card][dim], device, 16-byte aligned, caller-owned
 *   out        f32 [n_frames][dim], device, 16-byte aligned
 *   status     optional device word (e.g. the engine's); PP_S_INDEX is OR-ed into it
 *              when a code is >= card
 * A negative code (the -1 of a closed slot) adds nothing; a code >= card adds nothing.
 * 1 <= n_books <= 32, code_stride >= n_books, dim a positive multiple of 4; n_frames == 0
 * does nothing.  Asynchronous on `stream`.  Errors: PP_EINVAL, PP_E_CUDA. */
int pp_rvq_dequantize(const int32_t* codes, int code_stride, int n_frames, int n_books,
                      const float* codebooks, int card, int dim, float* out, uint32_t* status,
                      void* stream);

#ifdef __cplusplus
}
#endif
#endif
