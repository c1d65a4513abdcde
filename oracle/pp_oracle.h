/*
 * pp_oracle.h - CPU oracle of the PersonaPlex / Moshi 80 ms lockstep decode tick.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously-correct definition of
 * one tick of the RQ-Transformer that the CUDA path is checked against.  Only the
 * tests, the smoke check and the bench's CPU-baseline leg may load it; the product
 * library never does, and the two share no code, headers, tables or constants.
 *
 * Arithmetic: every activation, dot product, norm, softmax and RoPE rotation is in
 * fp64.  Weights are the given bf16 values (widened exactly); RMSNorm alphas are the
 * given fp32 values; the ring KV cache stores K and V rounded to bf16 (round to
 * nearest even), because the cache is a bf16 tensor (the full-window stress case fills
 * it with random bf16 values).  Logits are rounded to fp32 and the greedy decision
 * is taken on those fp32 values (the GPU kernel's precision), lowest index on ties,
 * NaN never chosen.  The sampling variants likewise take their decision steps (penalty,
 * temperature, expf) in fp32 and accumulate probability masses in fp64.
 *
 * Sources (page title, section):
 *  - vllm-omni recipes/NVIDIA/PersonaPlex.md, "Architecture": temporal 4096-d / 32
 *    layers / 32 heads with a 3000-frame sliding window in a per-slot ring KV cache;
 *    depformer 1024-d / 6 layers / 16 heads, autoregressive over 16 codebooks, reset
 *    each frame; the [B,17,1] column (row 0 text, rows 1-8 agent audio, rows 9-16
 *    user audio); persona and voice forced through the same step.
 *  - "PersonaPlex full-duplex ... vLLM-Omni 80ms Lockstep" (mhpq.cn), sections
 *    "架构" (fp32 RMSNorm alpha, fused in-proj attention, interleaved RoPE at the
 *    absolute position, SiLU-gated MLP), "帧 token 布局" (TEXT_INITIAL_TOKEN 32000,
 *    AUDIO_INITIAL_TOKEN 2048), "贪心解码与 Parity 约束" (greedy, relative-position
 *    causal mask), "运维要点" (_RingKV start-offset mask, recycled slot bit-exact).
 *
 * Readings where the pages are silent are stated at each function in pp_oracle.c.
 * Parity status of every function is pinned by tests/test_oracle_pins.py.
 */
#ifndef PP_ORACLE_H
#define PP_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t d, n_layers, n_heads, ffn;
  int32_t text_vocab;   /* text logits; the text table has text_vocab+1 rows */
  int32_t audio_card;   /* audio logits; each audio table has audio_card+1 rows */
  int32_t n_q;          /* 16 audio rows per column */
  int32_t dep_d, dep_layers, dep_heads, dep_ffn;
  int32_t window;
  double eps, rope_base;
} ora_shape;

/* Host pointers; matrices are row-major [out, in]; per-layer tensors are stacked. */
typedef struct {
  const uint16_t* emb_text;       /* [Vt+1, d] */
  const uint16_t* emb_audio;      /* [n_q, Va+1, d] */
  const float* attn_alpha;        /* [L, d] */
  const uint16_t* wqkv;           /* [L, 3d, d]   rows: q heads, k heads, v heads */
  const uint16_t* wo;             /* [L, d, d] */
  const float* mlp_alpha;         /* [L, d] */
  const uint16_t* wgu;            /* [L, 2F, d]   rows: gate (F), up (F) */
  const uint16_t* wdown;          /* [L, d, F] */
  const float* out_alpha;         /* [d] */
  const uint16_t* wtext;          /* [Vt, d] */
  const uint16_t* dep_inproj;     /* [n_q, dd, d] */
  const uint16_t* dep_emb_text;   /* [Vt+1, dd] */
  const uint16_t* dep_emb_audio;  /* [n_q-1, Va+1, dd] */
  const float* dep_attn_alpha;    /* [Ld, dd] */
  const uint16_t* dep_wqkv;       /* [Ld, 3dd, dd] */
  const uint16_t* dep_wo;         /* [Ld, dd, dd] */
  const float* dep_mlp_alpha;     /* [Ld, dd] */
  const uint16_t* dep_wgu;        /* [Ld, 2Fd, dd] */
  const uint16_t* dep_wdown;      /* [Ld, dd, Fd] */
  const float* dep_out_alpha;     /* [dd] */
  const uint16_t* dep_heads;      /* [n_q, Va, dd] */
} ora_weights;

/* One session: its ring (caller-owned) and absolute position (frames since open). */
typedef struct {
  uint16_t* ring_k;   /* [L, H, W, Dh] bf16 */
  uint16_t* ring_v;   /* [L, H, W, Dh] bf16 */
  int64_t pos;
} ora_session;

/* ---- building blocks (each pinned separately by the tests) ---------------------- */
double ora_bf16_to_f64(uint16_t b);
uint16_t ora_f64_to_bf16(double x);
void ora_rmsnorm(const double* x, const float* alpha, int n, double eps, double* y);
void ora_matvec(const uint16_t* w, int rows, int cols, const double* x, double* y);
void ora_rope(double* v, int n_heads, int head_dim, int64_t pos, double base);
void ora_ring_write(uint16_t* ring_head, int window, int head_dim, int64_t pos,
                    const double* kv);
void ora_attend(const double* q, const uint16_t* k_head, const uint16_t* v_head,
                int n_valid, int head_dim, double* out);
int32_t ora_argmax_f32(const float* v, int n);
void ora_embed(const ora_shape* s, const ora_weights* w, const int32_t* column, double* x);

/* ---- the tick ------------------------------------------------------------------- */
/* Temporal transformer for one session at its position: writes this frame's K/V into
 * the ring and returns z = RMSNorm(x_L) * out_alpha (length d).  Does not advance pos. */
void ora_temporal(const ora_shape* s, const ora_weights* w, ora_session* sess,
                  const int32_t* prev_column, double* z);
/* Text head: logits (fp32, length Vt) of z. */
void ora_text_head(const ora_shape* s, const ora_weights* w, const double* z, float* logits);
/* Depformer over the 16 codebook steps of one frame, from a fresh (reset) cache.
 * column[0] must hold this frame's text token; rows 1..16 are written.
 * logits: [n_q, Va] fp32 or NULL. */
void ora_depformer(const ora_shape* s, const ora_weights* w, const double* z,
                   const uint8_t* force_mask, const int32_t* forced,
                   const int32_t* user_codes, int32_t* column, float* logits);
/* One full tick: embed -> temporal -> text head (greedy or forced) -> depformer ->
 * pos += 1.  logits_text [Vt] and logits_audio [n_q, Va] may be NULL. */
/* Mimi RVQ dequantisation, the first step after the tick (mhpq section 2.3 "Mimi": 8
 * codebooks of 2048 entries at 12.5 Hz, residual vector quantisation; Recipe,
 * Architecture: each output column carries the agent's 8 audio codes).  A residual
 * quantiser's latent is the sum of the entries it selected, one per codebook:
 *   out[f][d] = sum_{k < n_books} codebooks[k][codes[f*code_stride + k]][d]
 * in fp64.  A negative code (the -1 a closed slot emits) adds nothing; a code >= card
 * adds nothing and is counted in *bad. */
void ora_rvq_dequantize(const int32_t* codes, int code_stride, int n_frames, int n_books,
                        const float* codebooks, int card, int dim, double* out, int* bad);

/* Sampling variants (the reading is stated at the definitions in pp_oracle.c).
 * ora_sample returns the token and, in alts[0 .. *n_alts), every token that the same
 * steps give when the draw's target moves by tol (relative to the kept mass) or the
 * nucleus cut moves by one run where its mass or value lies that close to the cut:
 * the decisions an fp32 evaluation of the steps may reach.  *n_kept counts the tokens
 * left after the filters. */
#define ORA_SAMPLE_MAX_ALTS 9
void ora_philox4x64(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]);
float ora_sample_uniform(uint64_t seed, int64_t pos, int row);
int32_t ora_sample(const float* logits, int n, float temperature, int top_k, float top_p,
                   float penalty, const int32_t* hist, int n_hist, float u, double tol,
                   int* n_kept, int32_t* alts, int* n_alts);

void ora_step(const ora_shape* s, const ora_weights* w, ora_session* sess,
              const int32_t* prev_column, const int32_t* user_codes,
              const uint8_t* force_mask, const int32_t* forced, int32_t* column,
              float* logits_text, float* logits_audio);

#ifdef __cplusplus
}
#endif
#endif
