"""The pins must catch plausible mistakes: each case below plants one mistake (one or
more edits of the same slip) in a temporary copy of the oracle source (never in the
committed file), rebuilds it, runs the pin suite against the copy in a subprocess and
expects a failure."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pp_oracle.c")

MUTANTS = {
    "drop_alpha": ("y[i] = x[i] * r * (double)alpha[i];", "y[i] = x[i] * r;"),
    "eps_outside_sqrt": ("1.0 / sqrt(ss / (double)n + eps)", "1.0 / (sqrt(ss / (double)n) + eps)"),
    "rope_sign": ("hv[2 * i] = a * c - b * sn;", "hv[2 * i] = a * c + b * sn;"),
    "rope_half_split": ("double a = hv[2 * i], b = hv[2 * i + 1];",
                        "double a = hv[i], b = hv[i + head_dim / 2];"),
    "window_excludes_current": ("const int n_valid = (int)(p + 1 < W ? p + 1 : W);",
                                "const int n_valid = (int)(p < W ? (p > 0 ? p : 1) : W);"),
    "ring_index_no_mod": ("(int64_t)(pos % window) * head_dim", "(int64_t)(pos % (window + 1) % window) * head_dim"),
    "kv_order_swapped": ("double* k = qkv + d;\n    double* v = qkv + 2 * d;",
                         "double* v = qkv + d;\n    double* k = qkv + 2 * d;"),
    "gate_up_swapped": ("h[i] = silu(gu[i]) * gu[F + i];", "h[i] = gu[i] * silu(gu[F + i]);"),
    "matvec_transposed": ("const uint16_t* wr = w + (int64_t)r * cols;\n    double acc = 0.0;\n    for (int c = 0; c < cols; ++c) acc += ora_bf16_to_f64(wr[c]) * x[c];",
                          "double acc = 0.0;\n    for (int c = 0; c < cols && c < rows; ++c) acc += ora_bf16_to_f64(w[(int64_t)c * cols + r]) * x[c];"),
    "attn_no_scale": ("s[j] = dot * scale;", "s[j] = dot;"),
    "audio_table_off_by_one": ("w->emb_audio + ((int64_t)(r - 1) * (s->audio_card + 1) + column[r]) * d;",
                               "w->emb_audio + ((int64_t)(r % s->n_q) * (s->audio_card + 1) + column[r]) * d;"),
    "dep_row_off_by_one": ("int row = k + 1;", "int row = k + (k < 15);"),
    "dep_no_reset_causal": ("for (int j = 0; j <= k; ++j) {\n          const double* kj",
                            "for (int j = 0; j <= k && j < 1; ++j) {\n          const double* kj"),
    "argmax_last_tie": ("if (best < 0 || v[i] > v[best]) best = i;", "if (best < 0 || v[i] >= v[best]) best = i;"),
    "rvq_wrong_book": ("const float* e = codebooks + ((size_t)k * card + c) * dim;",
                       "const float* e = codebooks + ((size_t)(k ? k - 1 : 0) * card + c) * dim;"),
    "rvq_skips_first_book": ("for (int k = 0; k < n_books; ++k) {\n      const int32_t c",
                             "for (int k = 1; k < n_books; ++k) {\n      const int32_t c"),
    "rvq_negative_counted": ("      if (c < 0) continue;\n", "      if (c < 0) {\n        ++nbad;\n        continue;\n      }\n"),
    "philox_key_bump_swapped": ("      k0 += W0;\n      k1 += W1;", "      k0 += W1;\n      k1 += W0;"),
    "philox_products_swapped": ("const uint64_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;",
                                "const uint64_t n0 = hi0 ^ c1 ^ k0, n1 = lo0, n2 = hi1 ^ c3 ^ k1, n3 = lo1;"),
    "uniform_low_bits": ("(float)(out[row % 4] >> 40)", "(float)(out[row % 4] & 0xFFFFFFu)"),
    "uniform_block_by_word": ("(uint64_t)(row / 4), 0, 0}", "(uint64_t)(row % 4), 0, 0}"),
    "temperature_multiplies": ("v[i] = v[i] / temperature;", "v[i] = v[i] * temperature;"),
    "penalty_unsigned": ("v[h] = v[h] > 0.f ? v[h] / penalty : v[h] * penalty;", "v[h] = v[h] / penalty;"),
    "penalty_per_occurrence": ("    if (seen) continue;\n", "    (void)seen;\n"),
    "top_k_off_by_one": ("tk = srt[top_k - 1];", "tk = srt[top_k];"),
    "nucleus_drops_the_cut": ("        tp = val;\n", "        tp = start > 0 ? srt[start - 1] : val;\n"),
    "cdf_not_strict": ("    if (run > target) return i;", "    if (run >= target) return i;"),
    "cdf_ignores_kept_set": ("    if (!(e[i] > 0.f && e[i] >= tp)) continue;\n", "    if (!(e[i] > 0.f)) continue;\n"),
    # the depformer's own MLP, step attention and per-frame cache
    "dep_gate_up_swapped": ("h[i] = silu(gu[i]) * gu[Fd + i];", "h[i] = gu[i] * silu(gu[Fd + i]);"),
    "dep_no_score_scale": ("sc[j] = dot / sqrt((double)Dhd);", "sc[j] = dot;"),
    "dep_scale_by_width": ("sc[j] = dot / sqrt((double)Dhd);", "sc[j] = dot / sqrt((double)dd);"),
    "dep_mlp_norm_wrong_alpha": ("ora_rmsnorm(y, w->dep_mlp_alpha + (int64_t)l * dd, dd, s->eps, n);",
                                 "ora_rmsnorm(y, w->dep_attn_alpha + (int64_t)l * dd, dd, s->eps, n);"),
    # the cache is made once (large enough for every test shape), never cleared, and
    # read over all of its 16 entries
    "dep_cache_carried_across_frames": [
        ("  double* kc = (double*)calloc((size_t)Ld * nq * dd, sizeof(double));\n"
         "  double* vc = (double*)calloc((size_t)Ld * nq * dd, sizeof(double));\n",
         "  static double* kc = 0;\n  static double* vc = 0;\n"
         "  if (!kc) kc = (double*)calloc((size_t)8 * 16 * 4096, sizeof(double));\n"
         "  if (!vc) vc = (double*)calloc((size_t)8 * 16 * 4096, sizeof(double));\n"),
        ("free(lg); free(lf); free(kc); free(vc); free(sc);", "free(lg); free(lf); free(sc);"),
        ("for (int j = 0; j <= k; ++j) {\n          const double* kj",
         "for (int j = 0; j < nq; ++j) {\n          const double* kj"),
        ("for (int j = 0; j <= k; ++j) { sc[j] = exp(sc[j] - m); lsum += sc[j]; }",
         "for (int j = 0; j < nq; ++j) { sc[j] = exp(sc[j] - m); lsum += sc[j]; }"),
        ("for (int j = 0; j <= k; ++j)\n            acc += sc[j]",
         "for (int j = 0; j < nq; ++j)\n            acc += sc[j]"),
    ],
}

# mistakes in the sampling variants, caught by their own pin file
SAMPLING = {"philox_key_bump_swapped", "philox_products_swapped", "uniform_low_bits",
            "uniform_block_by_word", "temperature_multiplies", "penalty_unsigned",
            "penalty_per_occurrence", "top_k_off_by_one", "nucleus_drops_the_cut",
            "cdf_not_strict", "cdf_ignores_kept_set"}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    edits = MUTANTS[name]
    if isinstance(edits, tuple):
        edits = [edits]
    src = open(SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, "mutation anchor not found: %s" % name
        src = src.replace(old, new)
    shutil.copy(os.path.join(ROOT, "oracle", "pp_oracle.h"), tmp_path / "pp_oracle.h")
    (tmp_path / "pp_oracle.c").write_text(src)
    so = str(tmp_path / "libmutant.so")
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                           "-std=c11", str(tmp_path / "pp_oracle.c"), "-o", so, "-lm"])
    env = dict(os.environ, PP_ORACLE_SO=so)
    pins = "test_oracle_sampling_pins.py" if name in SAMPLING else "test_oracle_pins.py"
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", pins)],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "planted mistake %s was not caught:\n%s" % (name, r.stdout[-2000:])
