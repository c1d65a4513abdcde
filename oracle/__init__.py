"""CPU oracle of the PersonaPlex / Moshi 80 ms lockstep decode tick.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke`` and the CPU-baseline
leg of ``bench.py`` use it to check and time the CUDA path.  It imports nothing from
the product package or its native library, and the product never imports it.

The arithmetic lives in ``pp_oracle.c`` (plain C, fp64, one function per step of the
tick, each citing the page section it follows).  This module only marshals numpy
arrays into it.  Shapes are read by attribute name from any object that has them
(``d``, ``n_layers``, ``n_heads``, ``ffn``, ``text_vocab``, ``audio_card``, ``n_q``,
``dep_d``, ``dep_layers``, ``dep_heads``, ``dep_ffn``, ``window``, ``eps``,
``rope_base``).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_SHAPE_FIELDS = ["d", "n_layers", "n_heads", "ffn", "text_vocab", "audio_card", "n_q",
                 "dep_d", "dep_layers", "dep_heads", "dep_ffn", "window"]
WEIGHT_FIELDS = ["emb_text", "emb_audio", "attn_alpha", "wqkv", "wo", "mlp_alpha", "wgu",
                 "wdown", "out_alpha", "wtext", "dep_inproj", "dep_emb_text", "dep_emb_audio",
                 "dep_attn_alpha", "dep_wqkv", "dep_wo", "dep_mlp_alpha", "dep_wgu",
                 "dep_wdown", "dep_out_alpha", "dep_heads"]


class OraShape(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int32) for f in _SHAPE_FIELDS] + [
        ("eps", ctypes.c_double), ("rope_base", ctypes.c_double)]


class OraWeights(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in WEIGHT_FIELDS]


class OraSession(ctypes.Structure):
    _fields_ = [("ring_k", ctypes.c_void_p), ("ring_v", ctypes.c_void_p),
                ("pos", ctypes.c_int64)]


def lib():
    global _lib
    if _lib is None:
        so = os.environ.get("PP_ORACLE_SO")   # a test may point at a rebuilt variant
        if not so:
            _build.build()
            so = _build.SO
        L = ctypes.CDLL(so)
        P = ctypes.c_void_p
        L.ora_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.ora_bf16_to_f64.restype = ctypes.c_double
        L.ora_f64_to_bf16.argtypes = [ctypes.c_double]
        L.ora_f64_to_bf16.restype = ctypes.c_uint16
        L.ora_rmsnorm.argtypes = [P, P, ctypes.c_int, ctypes.c_double, P]
        L.ora_matvec.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P]
        L.ora_rope.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_double]
        L.ora_ring_write.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int64, P]
        L.ora_attend.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, P]
        L.ora_argmax_f32.argtypes = [P, ctypes.c_int]
        L.ora_argmax_f32.restype = ctypes.c_int32
        L.ora_embed.argtypes = [P, P, P, P]
        L.ora_temporal.argtypes = [P, P, P, P, P]
        L.ora_text_head.argtypes = [P, P, P, P]
        L.ora_depformer.argtypes = [P, P, P, P, P, P, P, P]
        L.ora_step.argtypes = [P] * 10
        L.ora_rvq_dequantize.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                         ctypes.c_int, ctypes.c_int, P, P]
        L.ora_rvq_dequantize.restype = None
        L.ora_philox4x64.argtypes = [P, P, P]
        L.ora_philox4x64.restype = None
        L.ora_sample_uniform.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int]
        L.ora_sample_uniform.restype = ctypes.c_float
        L.ora_sample.argtypes = [P, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_float,
                                 ctypes.c_float, P, ctypes.c_int, ctypes.c_float,
                                 ctypes.c_double, P, P, P]
        L.ora_sample.restype = ctypes.c_int32
        _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


# ---- building blocks -------------------------------------------------------------

def bf16_to_f64(b):
    return lib().ora_bf16_to_f64(int(b))


def f64_to_bf16(x):
    return lib().ora_f64_to_bf16(float(x))


def rmsnorm(x, alpha, eps):
    x, px = _c(x, np.float64)
    a, pa = _c(alpha, np.float32)
    y = np.empty_like(x)
    lib().ora_rmsnorm(px, pa, x.size, eps, y.ctypes.data)
    return y


def matvec(w_bf16, x):
    w, pw = _c(w_bf16, np.uint16)
    x, px = _c(x, np.float64)
    y = np.empty(w.shape[0], dtype=np.float64)
    lib().ora_matvec(pw, w.shape[0], w.shape[1], px, y.ctypes.data)
    return y


def rope(v, n_heads, head_dim, pos, base):
    v = np.array(v, dtype=np.float64, copy=True)
    lib().ora_rope(v.ctypes.data, n_heads, head_dim, int(pos), float(base))
    return v


def ring_write(ring_head, pos, kv):
    """ring_head: uint16 [W, Dh] (modified in place)."""
    assert ring_head.flags.c_contiguous and ring_head.dtype == np.uint16
    kv, pk = _c(kv, np.float64)
    lib().ora_ring_write(ring_head.ctypes.data, ring_head.shape[0], ring_head.shape[1],
                         int(pos), pk)


def attend(q, k_head, v_head, n_valid):
    q, pq = _c(q, np.float64)
    k, pk = _c(k_head, np.uint16)
    v, pv = _c(v_head, np.uint16)
    out = np.empty(q.size, dtype=np.float64)
    lib().ora_attend(pq, pk, pv, int(n_valid), q.size, out.ctypes.data)
    return out


def argmax_f32(v):
    v, pv = _c(v, np.float32)
    return int(lib().ora_argmax_f32(pv, v.size))


# ---- the model -------------------------------------------------------------------

class Session:
    """One session's ring (bf16 [L, H, W, Dh] for K and V) and absolute position."""

    def __init__(self, shape, pos=0, ring_k=None, ring_v=None):
        s = shape
        dims = (s.n_layers, s.n_heads, s.window, s.d // s.n_heads)
        self.ring_k = np.zeros(dims, np.uint16) if ring_k is None else np.ascontiguousarray(
            ring_k, dtype=np.uint16)
        self.ring_v = np.zeros(dims, np.uint16) if ring_v is None else np.ascontiguousarray(
            ring_v, dtype=np.uint16)
        assert self.ring_k.shape == dims and self.ring_v.shape == dims
        self.c = OraSession(self.ring_k.ctypes.data, self.ring_v.ctypes.data, int(pos))

    @property
    def pos(self):
        return self.c.pos


class Oracle:
    """The tick on the CPU for one model (shape + host weights)."""

    def __init__(self, shape, weights):
        self.shape = shape
        self.cs = OraShape(*[int(getattr(shape, f)) for f in _SHAPE_FIELDS],
                           float(shape.eps), float(shape.rope_base))
        self._keep = {}
        ptrs = []
        for f in WEIGHT_FIELDS:
            dt = np.float32 if f.endswith("alpha") else np.uint16
            a = np.ascontiguousarray(weights[f], dtype=dt)
            self._keep[f] = a
            ptrs.append(a.ctypes.data)
        self.cw = OraWeights(*ptrs)

    def new_session(self, pos=0, ring_k=None, ring_v=None):
        return Session(self.shape, pos, ring_k, ring_v)

    def embed(self, column):
        col, pc = _c(column, np.int32)
        x = np.empty(self.shape.d, np.float64)
        lib().ora_embed(ctypes.byref(self.cs), ctypes.byref(self.cw), pc, x.ctypes.data)
        return x

    def temporal(self, sess, prev_column):
        col, pc = _c(prev_column, np.int32)
        z = np.empty(self.shape.d, np.float64)
        lib().ora_temporal(ctypes.byref(self.cs), ctypes.byref(self.cw), ctypes.byref(sess.c),
                           pc, z.ctypes.data)
        return z

    def text_head(self, z):
        z, pz = _c(z, np.float64)
        out = np.empty(self.shape.text_vocab, np.float32)
        lib().ora_text_head(ctypes.byref(self.cs), ctypes.byref(self.cw), pz, out.ctypes.data)
        return out

    def depformer(self, z, text_token, user_codes, force_mask=None, forced=None):
        s = self.shape
        z, pz = _c(z, np.float64)
        fm, pfm = _c(np.zeros(s.rows if hasattr(s, "rows") else 1 + s.n_q)
                     if force_mask is None else force_mask, np.uint8)
        ft, pft = _c(np.zeros(1 + s.n_q) if forced is None else forced, np.int32)
        uc, puc = _c(user_codes, np.int32)
        col = np.zeros(1 + s.n_q, np.int32)
        col[0] = text_token
        logits = np.empty((s.n_q, s.audio_card), np.float32)
        lib().ora_depformer(ctypes.byref(self.cs), ctypes.byref(self.cw), pz, pfm, pft, puc,
                            col.ctypes.data, logits.ctypes.data)
        return col, logits

    def step(self, sess, prev_column, user_codes, force_mask=None, forced=None,
             want_logits=True):
        """One tick; returns (column[17] int32, text logits [Vt] or None,
        audio logits [n_q, Va] or None)."""
        s = self.shape
        rows = 1 + s.n_q
        col_in, pc = _c(prev_column, np.int32)
        uc, puc = _c(user_codes, np.int32)
        fm, pfm = _c(np.zeros(rows) if force_mask is None else force_mask, np.uint8)
        ft, pft = _c(np.zeros(rows) if forced is None else forced, np.int32)
        col = np.zeros(rows, np.int32)
        lt = np.empty(s.text_vocab, np.float32) if want_logits else None
        la = np.empty((s.n_q, s.audio_card), np.float32) if want_logits else None
        lib().ora_step(ctypes.byref(self.cs), ctypes.byref(self.cw), ctypes.byref(sess.c),
                       pc, puc, pfm, pft, col.ctypes.data,
                       lt.ctypes.data if want_logits else None,
                       la.ctypes.data if want_logits else None)
        return col, lt, la


def rvq_dequantize(codes, codebooks, code_stride=None):
    """codes int32 [n, >= n_books] (row f's codes at f*code_stride), codebooks float32
    [n_books, card, dim] -> (latent float64 [n, dim], count of codes >= card)."""
    codes = np.ascontiguousarray(codes, dtype=np.int32)
    cb = np.ascontiguousarray(codebooks, dtype=np.float32)
    n_books, card, dim = cb.shape
    n = codes.shape[0]
    stride = codes.shape[1] if code_stride is None else code_stride
    out = np.empty((n, dim), dtype=np.float64)
    bad = ctypes.c_int(0)
    lib().ora_rvq_dequantize(codes.ctypes.data, stride, n, n_books, cb.ctypes.data, card, dim,
                             out.ctypes.data, ctypes.byref(bad))
    return out, bad.value


def philox4x64(counter, key):
    """Philox4x64-10 block: counter (4 x uint64), key (2 x uint64) -> 4 x uint64."""
    c = np.ascontiguousarray(counter, dtype=np.uint64)
    k = np.ascontiguousarray(key, dtype=np.uint64)
    out = np.empty(4, dtype=np.uint64)
    lib().ora_philox4x64(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def sample_uniform(seed, pos, row):
    """The uniform deciding row `row` (0 text, 1..8 agent audio) at session position pos."""
    return float(lib().ora_sample_uniform(int(seed) & (2**64 - 1), int(pos), int(row)))


# Relative distance to a decision boundary within which an fp32 evaluation may decide
# either way.  The GPU sums a row of <= 51200 non-negative terms as sequential chunks of
# <= 50 per thread, a 5-level warp scan or butterfly, an ordered sum of 32 warp totals
# and two more additions: relative error below (49 + 5 + 31 + 2) * 2^-24 = 5.2e-6; its
# expf and the oracle's differ by at most 3 ulp (3.6e-7 relative) per term.
SAMPLE_TOL = 6e-6


def sample(logits, u, temperature=1.0, top_k=0, top_p=1.0, penalty=1.0, history=(),
           tol=SAMPLE_TOL):
    """One sampled token from fp32 logits -> (token, alternatives, n_kept): the
    alternatives are every token the steps give with the target moved by tol or the
    nucleus cut moved by one run where that close (the token itself included)."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    h = np.ascontiguousarray(np.asarray(history, dtype=np.int32).reshape(-1))
    kept = ctypes.c_int(0)
    alts = np.zeros(9, np.int32)
    na = ctypes.c_int(0)
    t = lib().ora_sample(lg.ctypes.data, lg.size, float(temperature), int(top_k), float(top_p),
                         float(penalty), h.ctypes.data if h.size else None, int(h.size),
                         float(u), float(tol), ctypes.byref(kept), alts.ctypes.data,
                         ctypes.byref(na))
    return int(t), set(int(x) for x in alts[:na.value]), int(kept.value)


def initial_column(shape):
    """The column before the first frame: text initial token, then audio initial tokens
    (TEXT_INITIAL_TOKEN = text vocab size, AUDIO_INITIAL_TOKEN = codec cardinality)."""
    return np.array([shape.text_vocab] + [shape.audio_card] * shape.n_q, dtype=np.int32)
