"""Pins of the CPU oracle to things other than itself.

Each test ties one oracle function (or the wiring of the whole tick) to a closed
form, a library routine, a brute-force search or a structured-weight construction
whose answer is known in advance, so that a dropped term, a wrong sign or index, or
a transposed operand fails here before the oracle is trusted as the CUDA path's
reference.
"""
import dataclasses

import numpy as np
import pytest
import scipy.special

import oracle
import synth
from helpers import bf16_exact, bf16_rne_np, bf16_to_f64, perm_matrix, permutation

TINY = synth.TINY


# ---- number formats ------------------------------------------------------------------

def test_bf16_rounding_brute_force():
    """fp64 -> bf16 equals the nearest of all finite bf16 values (ties to even)."""
    pos = np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)
    vals = bf16_to_f64(pos)
    rng = np.random.default_rng(0)
    xs = list(np.ldexp(rng.uniform(0.5, 1.0, 3000), rng.integers(-140, 127, 3000)))
    mids = (vals[1:] + vals[:-1]) / 2.0            # exact ties
    xs += list(mids[rng.integers(0, mids.size, 2000)])
    xs += [np.nextafter(m, 0) for m in mids[rng.integers(0, mids.size, 500)]]
    xs += [np.nextafter(m, 1e300) for m in mids[rng.integers(0, mids.size, 500)]]
    for x in xs:
        i = np.searchsorted(vals, x)
        cands = [j for j in (i - 1, i) if 0 <= j < vals.size]
        best = min(cands, key=lambda j: (abs(vals[j] - x), int(pos[j]) & 1))
        assert oracle.f64_to_bf16(x) == pos[best], x
        assert oracle.f64_to_bf16(-x) == (pos[best] | 0x8000), x
    for u in rng.integers(0, 0x7F80, 2000):
        assert oracle.bf16_to_f64(int(u)) == bf16_to_f64(np.uint16(u))


# ---- RMSNorm -------------------------------------------------------------------------

def test_rmsnorm_closed_forms():
    n, eps = 64, 1e-5
    alpha = synth.normal_f32(n, 1, 1, 0.5) + np.float32(1)
    for c in [3.0, -0.25, 1e-3]:
        y = oracle.rmsnorm(np.full(n, c), alpha, eps)
        assert np.allclose(y, alpha.astype(np.float64) * c / np.sqrt(c * c + eps), rtol=1e-14)
    a, j = 2.5, 17
    x = np.zeros(n)
    x[j] = a
    y = oracle.rmsnorm(x, alpha, eps)
    expect = np.zeros(n)
    expect[j] = a / np.sqrt(a * a / n + eps) * alpha[j]
    assert np.allclose(y, expect, rtol=1e-14, atol=0)


# ---- matrix-vector product -----------------------------------------------------------

def test_matvec_matches_library_product():
    w = synth.normal_bf16(37 * 53, 2, 2, 0.02).reshape(37, 53)
    x = np.random.default_rng(1).standard_normal(53)
    y = oracle.matvec(w, x)
    assert np.allclose(y, bf16_to_f64(w) @ x, rtol=1e-12, atol=1e-15)
    # orientation: a permutation-selection matrix picks x entries
    src = permutation(53, 3)[:37]
    y = oracle.matvec(bf16_exact(perm_matrix(37, 53, src)), x)
    assert np.array_equal(y, x[src])


# ---- RoPE ----------------------------------------------------------------------------

def test_rope_is_complex_rotation():
    H, Dh, base = 3, 16, 10000.0
    rng = np.random.default_rng(2)
    v = rng.standard_normal(H * Dh)
    assert np.array_equal(oracle.rope(v, H, Dh, 0, base), v)     # position 0 is the identity
    for pos in [1, 7, 2999, 123456]:
        got = oracle.rope(v, H, Dh, pos, base).reshape(H, Dh // 2, 2)
        zc = v.reshape(H, Dh // 2, 2)
        zc = zc[..., 0] + 1j * zc[..., 1]
        freq = base ** (-2.0 * np.arange(Dh // 2) / Dh)
        rot = zc * np.exp(1j * pos * freq)
        assert np.allclose(got[..., 0], rot.real, atol=1e-12)
        assert np.allclose(got[..., 1], rot.imag, atol=1e-12)


def test_rope_relative_shift_invariance():
    Dh, base = 32, 10000.0
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(Dh), rng.standard_normal(Dh)
    ref = oracle.rope(q, 1, Dh, 40, base) @ oracle.rope(k, 1, Dh, 13, base)
    for shift in [1, 100, 5000]:
        got = oracle.rope(q, 1, Dh, 40 + shift, base) @ oracle.rope(k, 1, Dh, 13 + shift, base)
        assert abs(got - ref) < 1e-9 * max(1.0, abs(ref))


# ---- ring KV + attention ---------------------------------------------------------------

def _brute_attention(q, ks, vs, lo, hi):
    s = np.array([q @ ks[j] for j in range(lo, hi + 1)]) / np.sqrt(q.size)
    p = scipy.special.softmax(s)
    return p @ np.array(vs[lo:hi + 1])


@pytest.mark.parametrize("W", [1, 5, 8])
def test_ring_attention_equals_windowed_full_history(W):
    """Ring write at pos mod W + attention over min(pos+1, W) ring indices equals
    full attention over the last W absolute positions of the whole history."""
    Dh, T = 8, 3 * W + 4
    rng = np.random.default_rng(W)
    ring_k = np.zeros((W, Dh), np.uint16)
    ring_v = np.zeros((W, Dh), np.uint16)
    ks, vs = [], []
    for p in range(T):
        k, v = rng.standard_normal(Dh), rng.standard_normal(Dh)
        oracle.ring_write(ring_k, p, k)
        oracle.ring_write(ring_v, p, v)
        ks.append(bf16_to_f64(bf16_rne_np(k)))
        vs.append(bf16_to_f64(bf16_rne_np(v)))
        q = rng.standard_normal(Dh)
        got = oracle.attend(q, ring_k, ring_v, min(p + 1, W))
        ref = _brute_attention(q, ks, vs, max(0, p - W + 1), p)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_attention_special_cases():
    Dh = 16
    rng = np.random.default_rng(4)
    k = bf16_rne_np(rng.standard_normal((5, Dh)))
    v = bf16_rne_np(rng.standard_normal((5, Dh)))
    q = rng.standard_normal(Dh)
    # a single key returns its value exactly
    assert np.array_equal(oracle.attend(q, k, v, 1), bf16_to_f64(v[0]))
    # a zero query averages the values
    got = oracle.attend(np.zeros(Dh), k, v, 5)
    assert np.allclose(got, bf16_to_f64(v).mean(axis=0), rtol=1e-14, atol=1e-16)


# ---- greedy choice -------------------------------------------------------------------

def test_argmax_ties_and_nan():
    assert oracle.argmax_f32(np.array([1, 3, 3, 2], np.float32)) == 1
    assert oracle.argmax_f32(np.zeros(7, np.float32)) == 0
    assert oracle.argmax_f32(np.array([np.nan, 2, 5, np.nan, 5], np.float32)) == 2
    assert oracle.argmax_f32(np.array([-np.inf, -1e30], np.float32)) == 1
    assert oracle.argmax_f32(np.full(4, np.nan, np.float32)) == 0


# ---- embedding -----------------------------------------------------------------------

def _structured_tables(s):
    """Tables whose rows encode (table, row) exactly in bf16: text row t holds
    t & 255 in entry 2 and t >> 8 in entry 3; audio table a row c holds c & 255 in
    entry 8 + a and c >> 8 in entry 24 + a; every other entry is 0."""
    et = np.zeros((s.text_vocab + 1, s.d), np.float32)
    t = np.arange(s.text_vocab + 1)
    et[:, 2], et[:, 3] = t & 255, t >> 8
    ea = np.zeros((s.n_q, s.audio_card + 1, s.d), np.float32)
    c = np.arange(s.audio_card + 1)
    for a in range(s.n_q):
        ea[a, :, 8 + a], ea[a, :, 24 + a] = c & 255, c >> 8
    return bf16_exact(et), bf16_exact(ea)


def test_embed_row_mapping():
    s = TINY
    w = synth.make_weights_host(s, 0)
    w["emb_text"], w["emb_audio"] = _structured_tables(s)
    o = oracle.Oracle(s, w)
    col = synth.uniform_i32(17, 5, 5, 0, 2049)
    col[0] = 999
    x = o.embed(col)
    expect = np.zeros(s.d)
    expect[2], expect[3] = 999 & 255, 999 >> 8
    expect[8:24] = col[1:] & 255
    expect[24:40] = col[1:] >> 8
    assert np.array_equal(x, expect)


def test_embed_difference_is_exact():
    s = TINY
    w = synth.make_weights_host(s, 0)
    o = oracle.Oracle(s, w)
    base = oracle.initial_column(s)
    x0 = o.embed(base)
    for r, c in [(0, 17), (1, 5), (9, 2047), (16, 0)]:
        col = base.copy()
        col[r] = c
        diff = o.embed(col) - x0
        if r == 0:
            ref = bf16_to_f64(w["emb_text"][c]) - bf16_to_f64(w["emb_text"][base[0]])
        else:
            ref = bf16_to_f64(w["emb_audio"][r - 1, c]) - bf16_to_f64(w["emb_audio"][r - 1, base[r]])
        assert np.array_equal(diff, ref)


# ---- whole-tick wiring with structured weights ----------------------------------------

def _one_layer(s, window):
    return dataclasses.replace(s, n_layers=1, dep_layers=1, window=window)


def _zero(a):
    return np.zeros_like(a)


def _readout_text(s):
    """Text head [I_d; 0]: the first d text logits are fp32(z)."""
    wt = np.zeros((s.text_vocab, s.d), np.float32)
    wt[np.arange(s.d), np.arange(s.d)] = 1
    return bf16_exact(wt)


def _norm(x, a, eps):
    return x / np.sqrt(np.mean(x * x) + eps) * a.astype(np.float64)


def _embed_np(w, s, col):
    x = bf16_to_f64(w["emb_text"][col[0]])
    for r in range(1, 17):
        x = x + bf16_to_f64(w["emb_audio"][r - 1, col[r]])
    return x


def _columns(s, T, seed):
    cols = np.empty((T, 17), np.int32)
    cols[:, 0] = synth.uniform_i32(T, seed, 11, 0, s.text_vocab + 1)
    cols[:, 1:] = synth.uniform_i32(T * 16, seed, 12, 0, s.audio_card + 1).reshape(T, 16)
    return cols


def test_attention_value_path_window_and_out_projection():
    """q = k = 0, v = P_v n, W_o = P_o, MLP off: z_t = RMSNorm(x0_t + P_o mean_{window} bf16(v_j))."""
    s = _one_layer(TINY, 8)
    d = s.d
    w = synth.make_weights_host(s, 1, alpha="random")
    src_v, src_o = permutation(d, 10), permutation(d, 11)
    wqkv = np.zeros((1, 3 * d, d), np.float32)
    wqkv[0, 2 * d:] = perm_matrix(d, d, src_v)
    w["wqkv"] = bf16_exact(wqkv)
    w["wo"] = bf16_exact(perm_matrix(d, d, src_o)[None])
    w["wgu"], w["wdown"] = _zero(w["wgu"]), _zero(w["wdown"])
    w["wtext"] = _readout_text(s)
    o = oracle.Oracle(s, w)
    sess = o.new_session()
    cols = _columns(s, 21, 1)
    hist = []
    for t in range(21):
        _, lt, _ = o.step(sess, cols[t], np.zeros(8, np.int32))
        x0 = _embed_np(w, s, cols[t])
        v = _norm(x0, w["attn_alpha"][0], s.eps)[src_v]
        hist.append(bf16_to_f64(bf16_rne_np(v)))
        mean = np.mean(hist[max(0, t - s.window + 1):], axis=0)
        z = _norm(x0 + mean[src_o], w["out_alpha"], s.eps)
        assert np.allclose(lt[:d], z, rtol=2e-6, atol=1e-7), t


def test_mlp_gate_up_down_wiring():
    """Attention off; [g; u] = [P_g; P_u] n, W_down selects: x += (silu(g) * u)[src_d]."""
    s = _one_layer(TINY, 8)
    d, F = s.d, s.ffn
    w = synth.make_weights_host(s, 2, alpha="random")
    rng = np.random.default_rng(5)
    src_g, src_u = rng.integers(0, d, F), rng.integers(0, d, F)
    src_d = permutation(F, 12)[:d]
    w["wqkv"], w["wo"] = _zero(w["wqkv"]), _zero(w["wo"])
    w["wgu"] = bf16_exact(np.concatenate([perm_matrix(F, d, src_g), perm_matrix(F, d, src_u)])[None])
    w["wdown"] = bf16_exact(perm_matrix(d, F, src_d)[None])
    w["wtext"] = _readout_text(s)
    o = oracle.Oracle(s, w)
    sess = o.new_session()
    cols = _columns(s, 3, 2)
    for t in range(3):
        _, lt, _ = o.step(sess, cols[t], np.zeros(8, np.int32))
        x0 = _embed_np(w, s, cols[t])
        n = _norm(x0, w["mlp_alpha"][0], s.eps)
        g, u = n[src_g], n[src_u]
        h = g / (1 + np.exp(-g)) * u
        z = _norm(x0 + h[src_d], w["out_alpha"], s.eps)
        assert np.allclose(lt[:d], z, rtol=2e-6, atol=1e-7)


def _rope_np(v, H, Dh, pos, base):
    zc = v.reshape(H, Dh // 2, 2)
    zc = (zc[..., 0] + 1j * zc[..., 1]) * np.exp(1j * pos * base ** (-2.0 * np.arange(Dh // 2) / Dh))
    return np.stack([zc.real, zc.imag], axis=-1).reshape(-1)


def _brute_temporal(s, w, cols):
    """Numpy model of the temporal stack that keeps the FULL history of bf16 K/V per
    layer and applies the sliding window as an explicit position range."""
    d, H, Dh, F = s.d, s.n_heads, s.d // s.n_heads, s.ffn
    K = [[] for _ in range(s.n_layers)]
    V = [[] for _ in range(s.n_layers)]
    zs = []
    for t, col in enumerate(cols):
        x = _embed_np(w, s, col)
        for l in range(s.n_layers):
            n = _norm(x, w["attn_alpha"][l], s.eps)
            qkv = bf16_to_f64(w["wqkv"][l]) @ n
            q = _rope_np(qkv[:d], H, Dh, t, s.rope_base)
            k = _rope_np(qkv[d:2 * d], H, Dh, t, s.rope_base)
            K[l].append(bf16_to_f64(bf16_rne_np(k)).reshape(H, Dh))
            V[l].append(bf16_to_f64(bf16_rne_np(qkv[2 * d:])).reshape(H, Dh))
            lo = max(0, t - s.window + 1)
            att = np.concatenate([
                _brute_attention(q.reshape(H, Dh)[h], [kk[h] for kk in K[l]],
                                 [vv[h] for vv in V[l]], lo, t) for h in range(H)])
            x = x + bf16_to_f64(w["wo"][l]) @ att
            n = _norm(x, w["mlp_alpha"][l], s.eps)
            gu = bf16_to_f64(w["wgu"][l]) @ n
            g, u = gu[:F], gu[F:]
            x = x + bf16_to_f64(w["wdown"][l]) @ (g / (1 + np.exp(-g)) * u)
        zs.append(_norm(x, w["out_alpha"], s.eps))
    return zs


def test_temporal_equals_brute_force_full_attention():
    """Whole tiny temporal stack (random weights, ring wraps at W) against the
    full-history brute force."""
    s = dataclasses.replace(TINY, window=16)
    w = synth.make_weights_host(s, 3, alpha="random")
    # scale q/k rows up so that attention is far from uniform
    wq = bf16_to_f64(w["wqkv"]).copy()
    wq[:, :2 * s.d] *= 8.0
    w["wqkv"] = bf16_exact(wq.astype(np.float32))
    cols = _columns(s, 40, 3)
    ref = _brute_temporal(s, w, cols)
    o = oracle.Oracle(s, w)
    sess = o.new_session()
    for t in range(40):
        z = o.temporal(sess, cols[t])
        sess.c.pos += 1
        assert np.allclose(z, ref[t], rtol=1e-9, atol=1e-11), t


def test_text_head_and_forcing():
    s = TINY
    w = synth.make_weights_host(s, 4)
    o = oracle.Oracle(s, w)
    sess = o.new_session()
    col = oracle.initial_column(s)
    c1, lt, _ = o.step(sess, col, np.arange(8, dtype=np.int32))
    assert c1[0] == int(np.argmax(lt))
    assert np.array_equal(c1[9:], np.arange(8))
    fm = np.zeros(17, np.uint8)
    ft = np.zeros(17, np.int32)
    fm[0], ft[0] = 1, 123
    fm[4], ft[4] = 1, 77
    fm[12], ft[12] = 1, 5            # rows 9..16 always carry the user codes
    c2, _, _ = o.step(sess, col, np.arange(8, dtype=np.int32) + 100, fm, ft)
    assert c2[0] == 123 and c2[4] == 77 and c2[12] == 103


def _dep_structured(s, seed):
    """Depformer that maps a token to the next by a known rule: all layer weights 0,
    P_k = 0, D_k[tok] = one-hot at g(tok, k), H_k[c, dim] = 1 iff c = f(dim, k)."""
    dd, Va = s.dep_d, s.audio_card
    w = synth.make_weights_host(s, seed)
    for n in ["dep_wqkv", "dep_wo", "dep_wgu", "dep_wdown", "dep_inproj"]:
        w[n] = _zero(w[n])
    w["dep_out_alpha"] = np.ones(dd, np.float32)

    def g(tok, k):
        return (tok * 7 + 3 * k) % dd

    def f(dim, k):
        return (dim * 13 + 101 * k) % Va

    et = np.zeros((s.text_vocab + 1, dd), np.float32)
    et[np.arange(s.text_vocab + 1), g(np.arange(s.text_vocab + 1), 0)] = 1
    ea = np.zeros((s.n_q - 1, Va + 1, dd), np.float32)
    for k in range(1, s.n_q):
        ea[k - 1, np.arange(Va + 1), g(np.arange(Va + 1), k)] = 1
    hd = np.zeros((s.n_q, Va, dd), np.float32)
    for k in range(s.n_q):
        hd[k, f(np.arange(dd), k), np.arange(dd)] = 1
    w["dep_emb_text"], w["dep_emb_audio"], w["dep_heads"] = bf16_exact(et), bf16_exact(ea), bf16_exact(hd)
    return w, g, f


def test_depformer_row_chain_forcing_and_user_rows():
    s = TINY
    w, g, f = _dep_structured(s, 5)
    o = oracle.Oracle(s, w)
    uc = np.array([11, 22, 33, 44, 55, 66, 77, 88], np.int32)
    fm = np.zeros(17, np.uint8)
    ft = np.zeros(17, np.int32)
    fm[3], ft[3] = 1, 1500
    fm[8], ft[8] = 1, 9
    fm[10], ft[10] = 1, 4            # ignored: user row
    z = np.random.default_rng(6).standard_normal(s.d)
    col, _ = o.depformer(z, 421, uc, fm, ft)
    tok = 421
    for k in range(16):
        row = k + 1
        if row <= 8:
            nxt = ft[row] if fm[row] else f(g(tok, k), k)
        else:
            nxt = uc[row - 9]
        assert col[row] == nxt, row
        tok = nxt


def test_depformer_inproj_and_step_attention():
    """D = 0, P_k selects z entries, one layer with q = k = 0, v = n, W_o = P_o: the
    step-k state is e_k + P_o mean_{j<=k} RMSNorm(e_j), read through identity heads."""
    s = _one_layer(TINY, 8)
    d, dd = s.d, s.dep_d
    w = synth.make_weights_host(s, 6, alpha="random")
    w["dep_emb_text"], w["dep_emb_audio"] = _zero(w["dep_emb_text"]), _zero(w["dep_emb_audio"])
    srcs = [permutation(d, 20 + k)[:dd] for k in range(16)]
    w["dep_inproj"] = bf16_exact(np.stack([perm_matrix(dd, d, sk) for sk in srcs]))
    wqkv = np.zeros((1, 3 * dd, dd), np.float32)
    wqkv[0, 2 * dd:] = np.eye(dd)
    w["dep_wqkv"] = bf16_exact(wqkv)
    src_o = permutation(dd, 40)
    w["dep_wo"] = bf16_exact(perm_matrix(dd, dd, src_o)[None])
    w["dep_wgu"], w["dep_wdown"] = _zero(w["dep_wgu"]), _zero(w["dep_wdown"])
    heads = np.zeros((16, s.audio_card, dd), np.float32)
    heads[:, np.arange(dd), np.arange(dd)] = 1
    w["dep_heads"] = bf16_exact(heads)
    o = oracle.Oracle(s, w)
    z = np.random.default_rng(7).standard_normal(d)
    _, logits = o.depformer(z, 3, np.zeros(8, np.int32))
    ns = []
    for k in range(16):
        e = z[srcs[k]]
        ns.append(_norm(e, w["dep_attn_alpha"][0], s.eps))
        y = e + np.mean(ns, axis=0)[src_o]
        ref = _norm(y, w["dep_out_alpha"], s.eps)
        assert np.allclose(logits[k, :dd], ref, rtol=2e-6, atol=1e-7), k
        assert np.all(logits[k, dd:] == 0)


def _dep_identity_heads(s):
    heads = np.zeros((s.n_q, s.audio_card, s.dep_d), np.float32)
    heads[:, np.arange(s.dep_d), np.arange(s.dep_d)] = 1
    return bf16_exact(heads)


def test_depformer_mlp_gate_up_down_wiring():
    """Depformer attention off (W_qkv = W_o = 0), token tables 0, P_k selects z entries,
    [g; u] = [P_g; P_u] n with n = RMSNorm(e_k) * mlp_alpha (random), W_down selects:
    the step-k state is e_k + (silu(g) * u)[src_d], read through identity heads."""
    s = _one_layer(TINY, 8)
    d, dd, Fd = s.d, s.dep_d, s.dep_ffn
    w = synth.make_weights_host(s, 8, alpha="random")
    w["dep_emb_text"], w["dep_emb_audio"] = _zero(w["dep_emb_text"]), _zero(w["dep_emb_audio"])
    srcs = [permutation(d, 60 + k)[:dd] for k in range(16)]
    w["dep_inproj"] = bf16_exact(np.stack([perm_matrix(dd, d, sk) for sk in srcs]))
    w["dep_wqkv"], w["dep_wo"] = _zero(w["dep_wqkv"]), _zero(w["dep_wo"])
    rng = np.random.default_rng(61)
    src_g, src_u = rng.integers(0, dd, Fd), rng.integers(0, dd, Fd)
    src_d = permutation(Fd, 62)[:dd]
    w["dep_wgu"] = bf16_exact(np.concatenate([perm_matrix(Fd, dd, src_g),
                                              perm_matrix(Fd, dd, src_u)])[None])
    w["dep_wdown"] = bf16_exact(perm_matrix(dd, Fd, src_d)[None])
    w["dep_heads"] = _dep_identity_heads(s)
    o = oracle.Oracle(s, w)
    z = np.random.default_rng(63).standard_normal(d) * 2.0
    _, logits = o.depformer(z, 5, np.zeros(8, np.int32))
    for k in range(16):
        e = z[srcs[k]]
        n = _norm(e, w["dep_mlp_alpha"][0], s.eps)
        g, u = n[src_g], n[src_u]
        h = g / (1 + np.exp(-g)) * u
        ref = _norm(e + h[src_d], w["dep_out_alpha"], s.eps)
        assert np.allclose(logits[k, :dd], ref, rtol=2e-6, atol=1e-7), k


def _brute_depformer(s, w, z, tokens):
    """Numpy model of one frame's depformer as a single teacher-forced pass over all 16
    codebook positions at once: every position's input is known in advance (tokens[k]
    feeds step k), and causality is a -inf mask on the score matrix instead of a cache
    that grows step by step.  Returns the 16 heads' logits [16, Va] (fp64)."""
    dd, Hd, Fd, nq = s.dep_d, s.dep_heads, s.dep_ffn, s.n_q
    Dhd = dd // Hd
    X = np.empty((nq, dd))
    for k in range(nq):
        table = (bf16_to_f64(w["dep_emb_text"][tokens[0]]) if k == 0
                 else bf16_to_f64(w["dep_emb_audio"][k - 1, tokens[k]]))
        X[k] = bf16_to_f64(w["dep_inproj"][k]) @ z + table

    def norm_rows(A, alpha):
        return A / np.sqrt(np.mean(A * A, axis=1, keepdims=True) + s.eps) * alpha.astype(np.float64)

    mask = np.triu(np.full((nq, nq), -np.inf), 1)          # position i sees j <= i
    for l in range(s.dep_layers):
        N = norm_rows(X, w["dep_attn_alpha"][l])
        QKV = N @ bf16_to_f64(w["dep_wqkv"][l]).T
        Q, K, V = (QKV[:, i * dd:(i + 1) * dd].reshape(nq, Hd, Dhd) for i in range(3))
        S = np.einsum("ihc,jhc->hij", Q, K) / np.sqrt(Dhd) + mask
        P = scipy.special.softmax(S, axis=-1)
        O = np.einsum("hij,jhc->ihc", P, V).reshape(nq, dd)
        X = X + O @ bf16_to_f64(w["dep_wo"][l]).T
        N = norm_rows(X, w["dep_mlp_alpha"][l])
        GU = N @ bf16_to_f64(w["dep_wgu"][l]).T
        G, U = GU[:, :Fd], GU[:, Fd:]
        X = X + (scipy.special.expit(G) * G * U) @ bf16_to_f64(w["dep_wdown"][l]).T
    Zd = norm_rows(X, w["dep_out_alpha"])
    return np.stack([bf16_to_f64(w["dep_heads"][k]) @ Zd[k] for k in range(nq)])


def _scale_rows(wt, rows, factor):
    """bf16 weights with the given rows of every layer multiplied by a power of two."""
    v = bf16_to_f64(wt).copy()
    v[:, rows] *= factor
    return bf16_exact(v.astype(np.float32))


def test_depformer_equals_teacher_forced_causal_pass():
    """Random depformer weights (two layers, q and k rows scaled so the step attention is
    far from uniform), every agent row forced: the oracle's step-by-step decode with a
    per-frame cache equals one masked pass over the 16 known positions."""
    s = dataclasses.replace(TINY, dep_layers=2)
    dd = s.dep_d
    w = synth.make_weights_host(s, 9, alpha="random")
    w["dep_wqkv"] = _scale_rows(w["dep_wqkv"], slice(0, 2 * dd), 4.0)
    o = oracle.Oracle(s, w)
    rng = np.random.default_rng(64)
    for trial in range(3):
        z = rng.standard_normal(s.d)
        text = int(rng.integers(0, s.text_vocab + 1))
        agent = rng.integers(0, s.audio_card + 1, 8).astype(np.int32)
        user = rng.integers(0, s.audio_card, 8).astype(np.int32)
        fm = np.zeros(17, np.uint8)
        ft = np.zeros(17, np.int32)
        fm[1:9], ft[1:9] = 1, agent
        col, logits = o.depformer(z, text, user, fm, ft)
        assert np.array_equal(col[1:9], agent) and np.array_equal(col[9:], user)
        tokens = np.concatenate([[text], agent, user[:7]])
        ref = _brute_depformer(s, w, z, tokens)
        scale = np.abs(ref).max()
        assert np.allclose(logits, ref, rtol=1e-6, atol=1e-6 * scale), trial


def test_depformer_resets_every_frame():
    """The depformer's cache holds the current frame's steps only: each frame's rows 1..16
    and audio logits, taken in sequence through whole ticks, are bitwise those of the
    same frame's depformer run alone from its (z, text token, user codes), in order and
    in a shuffled order."""
    s = TINY
    w = synth.make_weights_host(s, 10, alpha="random")
    w["dep_wqkv"] = _scale_rows(w["dep_wqkv"], slice(0, 2 * s.dep_d), 4.0)
    o = oracle.Oracle(s, w)
    T = 6
    cols = _columns(s, T, 10)
    users = synth.uniform_i32(T * 8, 10, 13, 0, s.audio_card).reshape(T, 8)
    seq = o.new_session()
    rep = o.new_session()          # the same frames again, to read each frame's z
    frames = []
    for t in range(T):
        col, _, la = o.step(seq, cols[t], users[t])
        z = o.temporal(rep, cols[t])
        rep.c.pos += 1
        frames.append((z, int(col[0]), users[t], col, la))
    for order in (range(T), np.random.default_rng(11).permutation(T)):
        for t in order:
            z, text, user, col, la = frames[t]
            c2, l2 = o.depformer(z, text, user)
            assert np.array_equal(c2[1:], col[1:]), t
            assert np.array_equal(l2, la), t


# ---- Mimi RVQ dequantisation -----------------------------------------------------------

def _rvq_books(n_books=8, card=64, dim=16, seed=3):
    return np.random.default_rng(seed).standard_normal((n_books, card, dim)).astype(np.float32)


def test_rvq_single_codebook_returns_its_entry():
    """With every other code negative (no frame), the latent is exactly the one selected
    codebook entry."""
    cb = _rvq_books()
    for k in range(cb.shape[0]):
        codes = np.full((1, cb.shape[0]), -1, np.int32)
        codes[0, k] = 17
        out, bad = oracle.rvq_dequantize(codes, cb)
        assert bad == 0
        assert np.array_equal(out[0], cb[k, 17].astype(np.float64))


def test_rvq_is_additive_over_codebooks():
    """Dequantising codebooks {0..3} and {4..7} separately and adding gives the whole."""
    cb = _rvq_books()
    rng = np.random.default_rng(5)
    codes = rng.integers(0, cb.shape[1], size=(20, cb.shape[0]), dtype=np.int32)
    a, b = codes.copy(), codes.copy()
    a[:, 4:] = -1
    b[:, :4] = -1
    whole, _ = oracle.rvq_dequantize(codes, cb)
    pa, _ = oracle.rvq_dequantize(a, cb)
    pb, _ = oracle.rvq_dequantize(b, cb)
    assert np.allclose(whole, pa + pb, rtol=0, atol=1e-12)


def test_rvq_inverts_a_residual_encoder():
    """A greedy residual quantiser (each stage picks the entry nearest to what the
    previous stages left) encodes x; dequantising its codes gives x minus the final
    residual."""
    cb = _rvq_books(card=256, dim=8)
    x = np.random.default_rng(9).standard_normal((12, 8))
    codes = np.empty((12, cb.shape[0]), np.int32)
    r = x.copy()
    for k in range(cb.shape[0]):
        book = cb[k].astype(np.float64)
        d = ((r[:, None, :] - book[None, :, :]) ** 2).sum(-1)
        codes[:, k] = d.argmin(1)
        r = r - book[codes[:, k]]
    out, bad = oracle.rvq_dequantize(codes, cb)
    assert bad == 0
    assert np.allclose(out + r, x, rtol=0, atol=1e-12)
    assert np.linalg.norm(r) < np.linalg.norm(x)   # the stages did reduce the residual


def test_rvq_code_range():
    """Codes past the codebook add nothing and are counted; negative codes (a closed
    slot's -1 row) add nothing and are not."""
    cb = _rvq_books()
    col = np.random.default_rng(2).integers(0, cb.shape[1], size=(6, 17), dtype=np.int32)
    col[3, 1] = cb.shape[1]          # one code past the codebook
    col[4, 1:9] = -1                 # a closed slot's sentinel row
    out, bad = oracle.rvq_dequantize(col[:, 1:9], cb)
    assert bad == 1
    assert np.all(out[4] == 0)
    ref3 = sum(cb[k, col[3, 1 + k]].astype(np.float64) for k in range(1, 8))
    assert np.allclose(out[3], ref3, rtol=0, atol=1e-12)

