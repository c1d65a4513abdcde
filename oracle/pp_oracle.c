/*
 * pp_oracle.c - CPU oracle of the lockstep decode tick.  TEST INFRASTRUCTURE ONLY:
 * loaded by tests, the smoke check and the bench's CPU-baseline leg, never by the
 * product.  See pp_oracle.h for the arithmetic contract and the pages it follows.
 *
 * Style: plain loops in the order the definitions state them, fp64 throughout (the
 * sampling variants' fp32 decision steps excepted, see there),
 * OpenMP only across independent output rows of a matrix-vector product (each row's
 * dot product is one sequential loop), so results do not depend on the thread count.
 */
#include "pp_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- number formats ------------------------------------------------------------ */

double ora_bf16_to_f64(uint16_t b) {
  union { uint32_t u; float f; } v;
  v.u = (uint32_t)b << 16;
  return (double)v.f;
}

/* Round a double to the nearest bf16 (8 significant bits), ties to even, directly
 * from fp64 (no intermediate fp32 rounding).  Overflow gives +-inf. */
uint16_t ora_f64_to_bf16(double x) {
  union { uint32_t u; float f; } v;
  if (isnan(x)) return 0x7FC0;
  if (x == 0.0 || isinf(x)) {
    v.f = (float)x;
    return (uint16_t)(v.u >> 16);
  }
  int e;
  frexp(x, &e);                     /* |x| = m * 2^e, m in [0.5, 1) */
  int q = e - 8;                    /* quantum of an 8-bit significand */
  if (q < -133) q = -133;           /* bf16 subnormal quantum (same exponent range as fp32) */
  double r = nearbyint(ldexp(x, -q));  /* default rounding mode: to nearest, ties to even */
  double y = ldexp(r, q);
  if (fabs(y) > 3.3895313892515355e38) y = copysign(INFINITY, x);  /* above bf16 max */
  v.f = (float)y;                   /* exact: y has <= 8 significant bits */
  return (uint16_t)(v.u >> 16);
}

/* ---- building blocks ----------------------------------------------------------- */

/* RMSNorm with fp32 alpha ("fp32 RMSNorm alpha", 架构 section):
 *   y_i = x_i / sqrt(mean_j x_j^2 + eps) * alpha_i.
 * Reading: eps inside the square root, mean over the full width. */
void ora_rmsnorm(const double* x, const float* alpha, int n, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss / (double)n + eps);
  for (int i = 0; i < n; ++i) y[i] = x[i] * r * (double)alpha[i];
}

/* y = W x for a row-major bf16 W [rows, cols] (PyTorch Linear orientation, no bias). */
void ora_matvec(const uint16_t* w, int rows, int cols, const double* x, double* y) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    const uint16_t* wr = w + (int64_t)r * cols;
    double acc = 0.0;
    for (int c = 0; c < cols; ++c) acc += ora_bf16_to_f64(wr[c]) * x[c];
    y[r] = acc;
  }
}

/* Interleaved RoPE at absolute position pos ("交错 RoPE", 架构 section):
 * within each head, the pair (v[2i], v[2i+1]) is rotated by angle
 * pos * base^(-2i/head_dim).  Reading: base 10000, pos = frames since session open. */
void ora_rope(double* v, int n_heads, int head_dim, int64_t pos, double base) {
  for (int h = 0; h < n_heads; ++h) {
    double* hv = v + (int64_t)h * head_dim;
    for (int i = 0; i < head_dim / 2; ++i) {
      double theta = (double)pos * pow(base, -2.0 * (double)i / (double)head_dim);
      double c = cos(theta), sn = sin(theta);
      double a = hv[2 * i], b = hv[2 * i + 1];
      hv[2 * i] = a * c - b * sn;
      hv[2 * i + 1] = a * sn + b * c;
    }
  }
}

/* Ring KV write (_RingKV, 运维要点 section): the frame at absolute position pos goes to
 * ring index pos mod W, stored as bf16. */
void ora_ring_write(uint16_t* ring_head, int window, int head_dim, int64_t pos,
                    const double* kv) {
  uint16_t* dst = ring_head + (int64_t)(pos % window) * head_dim;
  for (int i = 0; i < head_dim; ++i) dst[i] = ora_f64_to_bf16(kv[i]);
}

/* Decode attention of one head over ring indices 0..n_valid-1:
 *   out = sum_j softmax_j(q . K_j / sqrt(Dh)) V_j.
 * With n_valid = min(pos+1, W) these indices hold exactly the absolute positions
 * max(0, pos-W+1)..pos (before the ring wraps they are 0..pos in place; after, every
 * index is live), i.e. the 3000-frame sliding window including the current frame.
 * Softmax is permutation invariant, so the ring order needs no un-rotation. */
void ora_attend(const double* q, const uint16_t* k_head, const uint16_t* v_head,
                int n_valid, int head_dim, double* out) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(n_valid > 0 ? n_valid : 1));
  double scale = 1.0 / sqrt((double)head_dim);
  double m = -INFINITY;
  for (int j = 0; j < n_valid; ++j) {
    const uint16_t* kj = k_head + (int64_t)j * head_dim;
    double dot = 0.0;
    for (int i = 0; i < head_dim; ++i) dot += q[i] * ora_bf16_to_f64(kj[i]);
    s[j] = dot * scale;
    if (s[j] > m) m = s[j];
  }
  double l = 0.0;
  for (int j = 0; j < n_valid; ++j) {
    s[j] = exp(s[j] - m);
    l += s[j];
  }
  for (int i = 0; i < head_dim; ++i) out[i] = 0.0;
  for (int j = 0; j < n_valid; ++j) {
    const uint16_t* vj = v_head + (int64_t)j * head_dim;
    for (int i = 0; i < head_dim; ++i) out[i] += s[j] * ora_bf16_to_f64(vj[i]);
  }
  if (n_valid > 0)
    for (int i = 0; i < head_dim; ++i) out[i] /= l;
  free(s);
}

/* Greedy choice on fp32 logits: the lowest index holding the maximum; NaN entries are
 * never chosen (all-NaN gives 0). */
int32_t ora_argmax_f32(const float* v, int n) {
  int32_t best = -1;
  for (int i = 0; i < n; ++i) {
    if (isnan(v[i])) continue;
    if (best < 0 || v[i] > v[best]) best = i;
  }
  return best < 0 ? 0 : best;
}

/* Input embedding of the previous column: the text table row of column[0] plus, for
 * r = 1..16, row column[r] of audio table r-1.  Tables have one extra row for the
 * initial token (TEXT_INITIAL_TOKEN = text vocab size, AUDIO_INITIAL_TOKEN = card). */
void ora_embed(const ora_shape* s, const ora_weights* w, const int32_t* column, double* x) {
  const int d = s->d;
  const uint16_t* t = w->emb_text + (int64_t)column[0] * d;
  for (int i = 0; i < d; ++i) x[i] = ora_bf16_to_f64(t[i]);
  for (int r = 1; r <= s->n_q; ++r) {
    const uint16_t* a =
        w->emb_audio + ((int64_t)(r - 1) * (s->audio_card + 1) + column[r]) * d;
    for (int i = 0; i < d; ++i) x[i] += ora_bf16_to_f64(a[i]);
  }
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* ---- temporal transformer ------------------------------------------------------ */

/* Helium temporal transformer, one frame of one session ("Temporal transformer",
 * Architecture).  Per layer: x += Wo Attn(RoPE(q), RoPE(k), v) with q,k,v = W_qkv
 * RMSNorm(x) (fused in-proj; reading: rows ordered q, k, v, heads contiguous, no
 * bias); then x += W_down (silu(g) * u) with [g; u] = W_gu RMSNorm(x) (reading: gate
 * rows first).  z = RMSNorm(x) * out_alpha. */
void ora_temporal(const ora_shape* s, const ora_weights* w, ora_session* sess,
                  const int32_t* prev_column, double* z) {
  const int d = s->d, H = s->n_heads, Dh = d / H, F = s->ffn, W = s->window;
  double* x = (double*)malloc(sizeof(double) * d);
  double* n = (double*)malloc(sizeof(double) * d);
  double* qkv = (double*)malloc(sizeof(double) * 3 * d);
  double* o = (double*)malloc(sizeof(double) * d);
  double* t = (double*)malloc(sizeof(double) * d);
  double* gu = (double*)malloc(sizeof(double) * 2 * F);
  double* h = (double*)malloc(sizeof(double) * F);
  const int64_t p = sess->pos;
  const int n_valid = (int)(p + 1 < W ? p + 1 : W);

  ora_embed(s, w, prev_column, x);
  for (int l = 0; l < s->n_layers; ++l) {
    ora_rmsnorm(x, w->attn_alpha + (int64_t)l * d, d, s->eps, n);
    ora_matvec(w->wqkv + (int64_t)l * 3 * d * d, 3 * d, d, n, qkv);
    double* q = qkv;
    double* k = qkv + d;
    double* v = qkv + 2 * d;
    ora_rope(q, H, Dh, p, s->rope_base);
    ora_rope(k, H, Dh, p, s->rope_base);
    for (int hh = 0; hh < H; ++hh) {
      int64_t base = ((int64_t)l * H + hh) * W * Dh;
      ora_ring_write(sess->ring_k + base, W, Dh, p, k + (int64_t)hh * Dh);
      ora_ring_write(sess->ring_v + base, W, Dh, p, v + (int64_t)hh * Dh);
    }
    for (int hh = 0; hh < H; ++hh) {
      int64_t base = ((int64_t)l * H + hh) * W * Dh;
      ora_attend(q + (int64_t)hh * Dh, sess->ring_k + base, sess->ring_v + base, n_valid, Dh,
                 o + (int64_t)hh * Dh);
    }
    ora_matvec(w->wo + (int64_t)l * d * d, d, d, o, t);
    for (int i = 0; i < d; ++i) x[i] += t[i];

    ora_rmsnorm(x, w->mlp_alpha + (int64_t)l * d, d, s->eps, n);
    ora_matvec(w->wgu + (int64_t)l * 2 * F * d, 2 * F, d, n, gu);
    for (int i = 0; i < F; ++i) h[i] = silu(gu[i]) * gu[F + i];
    ora_matvec(w->wdown + (int64_t)l * d * F, d, F, h, t);
    for (int i = 0; i < d; ++i) x[i] += t[i];
  }
  ora_rmsnorm(x, w->out_alpha, d, s->eps, z);
  free(x); free(n); free(qkv); free(o); free(t); free(gu); free(h);
}

void ora_text_head(const ora_shape* s, const ora_weights* w, const double* z, float* logits) {
  double* y = (double*)malloc(sizeof(double) * s->text_vocab);
  ora_matvec(w->wtext, s->text_vocab, s->d, z, y);
  for (int i = 0; i < s->text_vocab; ++i) logits[i] = (float)y[i];
  free(y);
}

/* ---- depformer ----------------------------------------------------------------- */

/* Depformer ("Depformer", Architecture): autoregressive over the 16 codebook steps
 * of one frame, with its own KV over the steps of this frame only (reset each frame).
 * Readings: step k's input is P_k z + D_k[tok_k], with tok_0 the frame's text token
 * (D_0 the depformer text table) and tok_k (k >= 1) the token already in row k (D_k
 * audio table k-1); the transformer layers are shared by all steps, causal over steps
 * 0..k, without positional encoding; a shared final RMSNorm feeds per-step heads H_k.
 * Step k decides row k+1: greedy (or forced) for agent rows 1..8, the incoming user
 * code for rows 9..16. */
void ora_depformer(const ora_shape* s, const ora_weights* w, const double* z,
                   const uint8_t* force_mask, const int32_t* forced,
                   const int32_t* user_codes, int32_t* column, float* logits) {
  const int d = s->d, dd = s->dep_d, Hd = s->dep_heads, Dhd = dd / Hd, Fd = s->dep_ffn;
  const int Ld = s->dep_layers, nq = s->n_q, Va = s->audio_card;
  double* y = (double*)malloc(sizeof(double) * dd);
  double* n = (double*)malloc(sizeof(double) * dd);
  double* qkv = (double*)malloc(sizeof(double) * 3 * dd);
  double* o = (double*)malloc(sizeof(double) * dd);
  double* t = (double*)malloc(sizeof(double) * dd);
  double* gu = (double*)malloc(sizeof(double) * 2 * Fd);
  double* h = (double*)malloc(sizeof(double) * Fd);
  double* zd = (double*)malloc(sizeof(double) * dd);
  double* lg = (double*)malloc(sizeof(double) * Va);
  float* lf = (float*)malloc(sizeof(float) * Va);
  /* this frame's depformer cache: [Ld][nq steps][dd], fresh for every frame */
  double* kc = (double*)calloc((size_t)Ld * nq * dd, sizeof(double));
  double* vc = (double*)calloc((size_t)Ld * nq * dd, sizeof(double));
  double* sc = (double*)malloc(sizeof(double) * nq);

  int32_t tok = column[0];
  for (int k = 0; k < nq; ++k) {
    ora_matvec(w->dep_inproj + (int64_t)k * dd * d, dd, d, z, y);
    const uint16_t* e = (k == 0)
        ? w->dep_emb_text + (int64_t)tok * dd
        : w->dep_emb_audio + ((int64_t)(k - 1) * (Va + 1) + tok) * dd;
    for (int i = 0; i < dd; ++i) y[i] += ora_bf16_to_f64(e[i]);

    for (int l = 0; l < Ld; ++l) {
      ora_rmsnorm(y, w->dep_attn_alpha + (int64_t)l * dd, dd, s->eps, n);
      ora_matvec(w->dep_wqkv + (int64_t)l * 3 * dd * dd, 3 * dd, dd, n, qkv);
      double* kl = kc + ((int64_t)l * nq + k) * dd;
      double* vl = vc + ((int64_t)l * nq + k) * dd;
      for (int i = 0; i < dd; ++i) { kl[i] = qkv[dd + i]; vl[i] = qkv[2 * dd + i]; }
      for (int hh = 0; hh < Hd; ++hh) {
        const double* qh = qkv + (int64_t)hh * Dhd;
        double m = -INFINITY, lsum = 0.0;
        for (int j = 0; j <= k; ++j) {
          const double* kj = kc + ((int64_t)l * nq + j) * dd + (int64_t)hh * Dhd;
          double dot = 0.0;
          for (int i = 0; i < Dhd; ++i) dot += qh[i] * kj[i];
          sc[j] = dot / sqrt((double)Dhd);
          if (sc[j] > m) m = sc[j];
        }
        for (int j = 0; j <= k; ++j) { sc[j] = exp(sc[j] - m); lsum += sc[j]; }
        for (int i = 0; i < Dhd; ++i) {
          double acc = 0.0;
          for (int j = 0; j <= k; ++j)
            acc += sc[j] * vc[((int64_t)l * nq + j) * dd + (int64_t)hh * Dhd + i];
          o[(int64_t)hh * Dhd + i] = acc / lsum;
        }
      }
      ora_matvec(w->dep_wo + (int64_t)l * dd * dd, dd, dd, o, t);
      for (int i = 0; i < dd; ++i) y[i] += t[i];
      ora_rmsnorm(y, w->dep_mlp_alpha + (int64_t)l * dd, dd, s->eps, n);
      ora_matvec(w->dep_wgu + (int64_t)l * 2 * Fd * dd, 2 * Fd, dd, n, gu);
      for (int i = 0; i < Fd; ++i) h[i] = silu(gu[i]) * gu[Fd + i];
      ora_matvec(w->dep_wdown + (int64_t)l * dd * Fd, dd, Fd, h, t);
      for (int i = 0; i < dd; ++i) y[i] += t[i];
    }
    ora_rmsnorm(y, w->dep_out_alpha, dd, s->eps, zd);
    ora_matvec(w->dep_heads + (int64_t)k * Va * dd, Va, dd, zd, lg);
    for (int i = 0; i < Va; ++i) lf[i] = (float)lg[i];
    if (logits) memcpy(logits + (int64_t)k * Va, lf, sizeof(float) * Va);

    int row = k + 1;
    if (row <= nq / 2)
      tok = force_mask[row] ? forced[row] : ora_argmax_f32(lf, Va);
    else
      tok = user_codes[row - 1 - nq / 2];
    column[row] = tok;
  }
  free(y); free(n); free(qkv); free(o); free(t); free(gu); free(h); free(zd);
  free(lg); free(lf); free(kc); free(vc); free(sc);
}

/* ---- one tick ------------------------------------------------------------------ */

void ora_step(const ora_shape* s, const ora_weights* w, ora_session* sess,
              const int32_t* prev_column, const int32_t* user_codes,
              const uint8_t* force_mask, const int32_t* forced, int32_t* column,
              float* logits_text, float* logits_audio) {
  double* z = (double*)malloc(sizeof(double) * s->d);
  float* lt = (float*)malloc(sizeof(float) * s->text_vocab);
  ora_temporal(s, w, sess, prev_column, z);
  ora_text_head(s, w, z, lt);
  column[0] = force_mask[0] ? forced[0] : ora_argmax_f32(lt, s->text_vocab);
  if (logits_text) memcpy(logits_text, lt, sizeof(float) * s->text_vocab);
  ora_depformer(s, w, z, force_mask, forced, user_codes, column, logits_audio);
  sess->pos += 1;
  free(z);
  free(lt);
}

/* ---- Mimi RVQ dequantisation --------------------------------------------------------- */

void ora_rvq_dequantize(const int32_t* codes, int code_stride, int n_frames, int n_books,
                        const float* codebooks, int card, int dim, double* out, int* bad) {
  int nbad = 0;
  for (int f = 0; f < n_frames; ++f) {
    double* o = out + (size_t)f * dim;
    for (int d = 0; d < dim; ++d) o[d] = 0.0;
    for (int k = 0; k < n_books; ++k) {
      const int32_t c = codes[(size_t)f * code_stride + k];
      if (c < 0) continue;
      if (c >= card) {
        ++nbad;
        continue;
      }
      const float* e = codebooks + ((size_t)k * card + c) * dim;
      for (int d = 0; d < dim; ++d) o[d] += (double)e[d];
    }
  }
  if (bad) *bad = nbad;
}

/* ---- sampling variants ------------------------------------------------------------
 *
 * The pages decode greedily and list the knobs a deployment may turn instead:
 * temperature, nucleus (top-p), repetition penalty and a separate audio temperature
 * ("PersonaPlex ... vLLM-Omni", deployment config; the persona-tuning article,
 * "generation parameters" and "repetition penalty").  They define none of the steps,
 * so the reading below is the plainest one that these knobs support, in this order:
 *   1. repetition penalty on the raw logits, in the signed form of Keskar et al.
 *      (CTRL, 2019) as commonly applied: each distinct token of the given history has
 *      its logit divided by R when positive and multiplied by R otherwise;
 *   2. division by the temperature;
 *   3. top-k: keep the logits at or above the k-th largest (ties at it are kept);
 *   4. e_i = exp(v_i - max v) over the kept logits;
 *   5. nucleus: the threshold is the largest e value whose own mass plus the mass of
 *      every larger e reaches p * sum(e); keep e at or above it (ties kept);
 *   6. inverse CDF in index order: the first kept index whose running mass exceeds
 *      u * (kept mass), else the last kept index.
 * Logits that are not finite are never chosen; with nothing left the token is 0.
 * Steps 1-4 are taken in fp32 (the decision's precision on the GPU: one IEEE
 * division or product per step, then expf), masses are accumulated in fp64.
 */

/* Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 * 1, 2, 3", SC 2011): ten rounds of two 64x64->128 multiplications with the published
 * multipliers, the key bumped by the published Weyl constants between rounds. */
void ora_philox4x64(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
  uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint64_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += W0;
      k1 += W1;
    }
    const unsigned __int128 p0 = (unsigned __int128)M0 * c0;
    const unsigned __int128 p1 = (unsigned __int128)M1 * c2;
    const uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
    const uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
    const uint64_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The uniform that decides row r (0 text, 1..8 agent audio) of the tick at session
 * position pos: word r % 4 of the Philox block at counter (pos, r / 4, 0, 0) under the
 * key (seed, 0), its top 24 bits scaled by 2^-24 (exact in fp32, in [0, 1)). */
float ora_sample_uniform(uint64_t seed, int64_t pos, int row) {
  const uint64_t ctr[4] = {(uint64_t)pos, (uint64_t)(row / 4), 0, 0};
  const uint64_t key[2] = {seed, 0};
  uint64_t out[4];
  ora_philox4x64(ctr, key, out);
  return (float)(out[row % 4] >> 40) * (1.0f / 16777216.0f);
}

static int cmp_f32_desc(const void* a, const void* b) {
  const float x = *(const float*)a, y = *(const float*)b;
  return (x < y) - (x > y);
}

/* Step 6 for one threshold: the first index e >= tp (e > 0) whose running mass
 * exceeds (u + shift) * (kept mass), else the last such index (-1: none). */
static int32_t inverse_cdf(const float* e, int n, float tp, double u, double shift) {
  double ZK = 0.0;
  int last = -1;
  for (int i = 0; i < n; ++i)
    if (e[i] > 0.f && e[i] >= tp) {
      ZK += (double)e[i];
      last = i;
    }
  const double target = (u + shift) * ZK;
  double run = 0.0;
  for (int i = 0; i < n; ++i) {
    if (!(e[i] > 0.f && e[i] >= tp)) continue;
    run += (double)e[i];
    if (run > target) return i;
  }
  return last;
}

static void add_alt(int32_t tok, int32_t* alts, int* n_alts) {
  for (int i = 0; i < *n_alts; ++i)
    if (alts[i] == tok) return;
  if (*n_alts < ORA_SAMPLE_MAX_ALTS) alts[(*n_alts)++] = tok;
}

int32_t ora_sample(const float* logits, int n, float temperature, int top_k, float top_p,
                   float penalty, const int32_t* hist, int n_hist, float u, double tol,
                   int* n_kept, int32_t* alts, int* n_alts) {
  float* v = (float*)malloc(sizeof(float) * (n > 0 ? n : 1));
  float* e = (float*)malloc(sizeof(float) * (n > 0 ? n : 1));
  float* srt = (float*)malloc(sizeof(float) * (n > 0 ? n : 1));
  int na = 0;
  int32_t alt_buf[ORA_SAMPLE_MAX_ALTS];
  for (int i = 0; i < n; ++i) v[i] = logits[i];
  /* 1. repetition penalty, once per distinct history token */
  for (int j = 0; j < n_hist; ++j) {
    const int32_t h = hist[j];
    if (h < 0 || h >= n) continue;
    int seen = 0;
    for (int i = 0; i < j; ++i) seen |= (hist[i] == h);
    if (seen) continue;
    v[h] = v[h] > 0.f ? v[h] / penalty : v[h] * penalty;
  }
  /* 2. temperature */
  int n_fin = 0;
  float m = -INFINITY;
  for (int i = 0; i < n; ++i) {
    v[i] = v[i] / temperature;
    if (isfinite(v[i])) {
      srt[n_fin++] = v[i];
      if (v[i] > m) m = v[i];
    }
  }
  if (n_fin == 0) {
    free(v); free(e); free(srt);
    if (n_kept) *n_kept = 0;
    if (n_alts) *n_alts = 1;
    if (alts) alts[0] = 0;
    return 0;
  }
  /* 3. top-k threshold: the k-th largest finite value */
  float tk = -INFINITY;
  if (top_k > 0 && top_k < n_fin) {
    qsort(srt, (size_t)n_fin, sizeof(float), cmp_f32_desc);
    tk = srt[top_k - 1];
  }
  /* 4. exponentials against the maximum */
  double Z = 0.0;
  for (int i = 0; i < n; ++i) {
    e[i] = (isfinite(v[i]) && v[i] >= tk) ? expf(v[i] - m) : 0.f;
    Z += (double)e[i];
  }
  /* 5. nucleus threshold: walk the e values from the largest down, a run of equal
   * values at a time, until the mass reaches p * Z.  Near the cut the GPU's fp32
   * masses (relative error below tol) or its expf (a few ulp, below 1e-6 relative)
   * may cut one run earlier or later: those thresholds are kept as alternatives. */
  float tp = 0.f, tp_alt[2] = {-1.f, -1.f};
  if (top_p < 1.f) {
    int ne = 0;
    for (int i = 0; i < n; ++i)
      if (e[i] > 0.f) srt[ne++] = e[i];
    qsort(srt, (size_t)ne, sizeof(float), cmp_f32_desc);
    const double P = (double)top_p * Z;
    double mass = 0.0;
    int j = 0;
    while (j < ne) {
      const int start = j;
      const float val = srt[j];
      const double before = mass;
      while (j < ne && srt[j] == val) mass += (double)srt[j++];
      if (mass >= P) {
        tp = val;
        if (j < ne && (mass - P < tol * Z || (double)srt[j] >= (double)val * (1.0 - 1e-6)))
          tp_alt[0] = srt[j];                          /* one run later */
        if (start > 0 && (P - before < tol * Z || (double)srt[start - 1] <= (double)val * (1.0 + 1e-6)))
          tp_alt[1] = srt[start - 1];                  /* one run earlier */
        break;
      }
    }
  }
  /* 6. inverse CDF in index order over the kept set */
  const int32_t tok = inverse_cdf(e, n, tp, (double)u, 0.0);
  add_alt(tok, alt_buf, &na);
  add_alt(inverse_cdf(e, n, tp, (double)u, -tol), alt_buf, &na);
  add_alt(inverse_cdf(e, n, tp, (double)u, tol), alt_buf, &na);
  for (int a = 0; a < 2; ++a)
    if (tp_alt[a] >= 0.f)
      for (int d = -1; d <= 1; ++d) add_alt(inverse_cdf(e, n, tp_alt[a], (double)u, d * tol), alt_buf, &na);
  int kept = 0;
  for (int i = 0; i < n; ++i) kept += (e[i] > 0.f && e[i] >= tp);
  free(v); free(e); free(srt);
  if (n_kept) *n_kept = kept;
  if (alts)
    for (int i = 0; i < na; ++i) alts[i] = alt_buf[i] < 0 ? 0 : alt_buf[i];
  if (n_alts) *n_alts = na;
  return tok < 0 ? 0 : tok;
}
