"""Seeded synthetic inputs for the PersonaPlex / Moshi lockstep tick.

No trained checkpoint, voice prompt, tokenizer or Mimi codes exist here, so every
input of the tick is drawn from a counter-based generator (Philox4x32-10, Salmon et
al. 2011) with the shapes and value distributions the workloads name:

* weights: bf16, N(0, 0.02) (8-term Irwin-Hall approximation), RMSNorm alpha fp32;
* ring KV for the full-window stress case: bf16 N(0, 1), counter = (slot, layer,
  K/V, element);
* token streams: uniform codes, forced prefill schedules, elastic join/leave events.

This module holds none of the tick's arithmetic.  Tests, ``bench.py`` and
``__graft_entry__.smoke`` call it to build identical inputs for the CPU oracle and
the CUDA path.
"""
import ctypes
import dataclasses
import os

import numpy as np

from . import build as _build

HERE = os.path.dirname(os.path.abspath(__file__))


@dataclasses.dataclass(frozen=True)
class Shape:
    """Model dimensions of one RQ-Transformer (temporal + depformer)."""
    d: int
    n_layers: int
    n_heads: int
    ffn: int
    text_vocab: int          # text logits; the text table has one more row (initial token)
    audio_card: int          # audio logits; each audio table has one more row
    n_q: int                 # audio rows of a column (8 agent + 8 user)
    dep_d: int
    dep_layers: int
    dep_heads: int
    dep_ffn: int
    window: int
    eps: float = 1e-5
    rope_base: float = 10000.0

    @property
    def head_dim(self):
        return self.d // self.n_heads

    @property
    def dep_head_dim(self):
        return self.dep_d // self.dep_heads

    @property
    def rows(self):
        return 1 + self.n_q


# The tiny bring-up model (256-d, 2 layers, 4 heads, FFN 704, text vocab 1000,
# depformer 128-d / 1 layer / 4 heads, window 64).
TINY = Shape(d=256, n_layers=2, n_heads=4, ffn=704, text_vocab=1000, audio_card=2048,
             n_q=16, dep_d=128, dep_layers=1, dep_heads=4, dep_ffn=352, window=64)
# A mid-size model with the full model's head dims (128 temporal, 64 depformer) and
# ragged tile counts, for parity at sizes the oracle still finishes in seconds.
SMALL = Shape(d=512, n_layers=2, n_heads=4, ffn=1408, text_vocab=1000, audio_card=2048,
              n_q=16, dep_d=256, dep_layers=2, dep_heads=4, dep_ffn=704, window=80)
# PersonaPlex-7B: Helium temporal 4096-d / 32 layers / 32 heads / FFN 11008, text vocab
# 32000, 16 audio tables of 2049 rows, depformer 1024-d / 6 layers / 16 heads, window 3000.
FULL = Shape(d=4096, n_layers=32, n_heads=32, ffn=11008, text_vocab=32000, audio_card=2048,
             n_q=16, dep_d=1024, dep_layers=6, dep_heads=16, dep_ffn=2816, window=3000)

PRESETS = {"tiny": TINY, "small": SMALL, "full": FULL}

BF16 = "bf16"
F32 = "f32"


def weight_specs(s):
    """(name, shape, dtype, stream id) of every weight tensor, stacked over layers."""
    d, L, F, dd, Ld, Fd = s.d, s.n_layers, s.ffn, s.dep_d, s.dep_layers, s.dep_ffn
    specs = [
        ("emb_text", (s.text_vocab + 1, d), BF16),
        ("emb_audio", (s.n_q, s.audio_card + 1, d), BF16),
        ("attn_alpha", (L, d), F32),
        ("wqkv", (L, 3 * d, d), BF16),
        ("wo", (L, d, d), BF16),
        ("mlp_alpha", (L, d), F32),
        ("wgu", (L, 2 * F, d), BF16),
        ("wdown", (L, d, F), BF16),
        ("out_alpha", (d,), F32),
        ("wtext", (s.text_vocab, d), BF16),
        ("dep_inproj", (s.n_q, dd, d), BF16),
        ("dep_emb_text", (s.text_vocab + 1, dd), BF16),
        ("dep_emb_audio", (s.n_q - 1, s.audio_card + 1, dd), BF16),
        ("dep_attn_alpha", (Ld, dd), F32),
        ("dep_wqkv", (Ld, 3 * dd, dd), BF16),
        ("dep_wo", (Ld, dd, dd), BF16),
        ("dep_mlp_alpha", (Ld, dd), F32),
        ("dep_wgu", (Ld, 2 * Fd, dd), BF16),
        ("dep_wdown", (Ld, dd, Fd), BF16),
        ("dep_out_alpha", (dd,), F32),
        ("dep_heads", (s.n_q, s.audio_card, dd), BF16),
    ]
    return [(n, shp, dt, 1 + i) for i, (n, shp, dt) in enumerate(specs)]


def weight_names():
    return [n for n, _, _, _ in weight_specs(TINY)]


# ---------------------------------------------------------------------------------
# native libraries
_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        _build.build(host=True, device=False)
        lib = ctypes.CDLL(_build.HOST_SO)
        lib.ppsyn_philox.argtypes = [ctypes.c_void_p] * 3
        lib.ppsyn_normal_scale.argtypes = [ctypes.c_double]
        lib.ppsyn_normal_scale.restype = ctypes.c_float
        lib.ppsyn_normal_bf16_host.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_uint32, ctypes.c_uint32, ctypes.c_float]
        lib.ppsyn_normal_f32_host.argtypes = lib.ppsyn_normal_bf16_host.argtypes
        lib.ppsyn_uniform_i32_host.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int32,
                                               ctypes.c_int32]
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        _build.build(host=False, device=True)
        lib = ctypes.CDLL(_build.DEV_SO)
        lib.ppsyn_normal_bf16_dev.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                              ctypes.c_uint32, ctypes.c_uint32, ctypes.c_float,
                                              ctypes.c_void_p]
        lib.ppsyn_normal_bf16_dev.restype = ctypes.c_int
        lib.ppsyn_normal_bf16_dev_blocks.argtypes = [
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_uint32, ctypes.c_uint32, ctypes.c_float, ctypes.c_void_p]
        lib.ppsyn_normal_bf16_dev_blocks.restype = ctypes.c_int
        _dev = lib
    return _dev


def philox(ctr, key):
    """One Philox4x32-10 block (for known-answer checks)."""
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _host_lib().ppsyn_philox(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def normal_scale(sigma):
    return _host_lib().ppsyn_normal_scale(float(sigma))


def normal_bf16(n, seed, stream, sigma, i0=0):
    """n bf16 N(0, sigma) deviates as uint16 bit patterns (host)."""
    out = np.empty(int(n), dtype=np.uint16)
    _host_lib().ppsyn_normal_bf16_host(out.ctypes.data, int(n), int(i0), seed, stream,
                                       normal_scale(sigma))
    return out


def normal_f32(n, seed, stream, sigma, i0=0):
    out = np.empty(int(n), dtype=np.float32)
    _host_lib().ppsyn_normal_f32_host(out.ctypes.data, int(n), int(i0), seed, stream,
                                      normal_scale(sigma))
    return out


def uniform_i32(n, seed, stream, lo, hi, i0=0):
    """n integers uniform in [lo, hi) (host)."""
    out = np.empty(int(n), dtype=np.int32)
    _host_lib().ppsyn_uniform_i32_host(out.ctypes.data, int(n), int(i0), seed, stream,
                                       int(lo), int(hi))
    return out


def bf16_to_f32(u16):
    """Widen bf16 bit patterns (uint16) to fp32 exactly."""
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


WEIGHT_SIGMA = 0.02
ALPHA_SIGMA = 0.25


def _alpha(shape, seed, stream, mode):
    n = int(np.prod(shape))
    if mode == "ones":
        return np.ones(shape, dtype=np.float32)
    # "random": 1 + N(0, 0.25) in fp32, to catch a kernel that drops alpha
    return (np.float32(1.0) + normal_f32(n, seed, stream, ALPHA_SIGMA)).reshape(shape)


def make_weights_host(s, seed, alpha="ones", names=None):
    """All weights of shape ``s`` as host numpy arrays (bf16 as uint16, alpha fp32)."""
    out = {}
    for name, shp, dt, stream in weight_specs(s):
        if names is not None and name not in names:
            continue
        if dt == F32:
            out[name] = _alpha(shp, seed, stream, alpha)
        else:
            out[name] = normal_bf16(int(np.prod(shp)), seed, stream, WEIGHT_SIGMA).reshape(shp)
    return out


def make_weights_device(s, seed, alpha="ones", device="cuda"):
    """The same weights as ``make_weights_host``, generated on the GPU (torch tensors).

    bf16 tensors are returned as torch.int16 storage holding the bf16 bit patterns."""
    import torch
    lib = _dev_lib()
    out = {}
    stream = torch.cuda.current_stream().cuda_stream
    for name, shp, dt, sid in weight_specs(s):
        if dt == F32:
            out[name] = torch.from_numpy(_alpha(shp, seed, sid, alpha)).to(device)
        else:
            t = torch.empty(shp, dtype=torch.int16, device=device)
            rc = lib.ppsyn_normal_bf16_dev(t.data_ptr(), t.numel(), 0, seed, sid,
                                           normal_scale(WEIGHT_SIGMA), stream)
            if rc != 0:
                raise RuntimeError("device weight fill failed: cuda error %d" % rc)
            out[name] = t
    return out


# ring KV fill for the full-window stress case ------------------------------------
KV_STREAM_BASE = 0x4B560000  # stream id of (slot, layer, k/v) = base + (slot*L + layer)*2 + kv
KV_SIGMA = 1.0


def kv_stream(slot, layer, kv, n_layers):
    return KV_STREAM_BASE + (slot * n_layers + layer) * 2 + kv


def ring_kv_host(s, seed, slot, layer, kv):
    """One (slot, layer, K or V) ring block [H, W, Dh] of bf16 N(0,1) deviates."""
    n = s.n_heads * s.window * s.head_dim
    v = normal_bf16(n, seed, kv_stream(slot, layer, kv, s.n_layers), KV_SIGMA)
    return v.reshape(s.n_heads, s.window, s.head_dim)


def ring_kv_fill_device(ptr, s, seed, slot, layer, kv, cuda_stream):
    """Fill the device ring block at ``ptr`` ([H, W, Dh] bf16, contiguous)."""
    n = s.n_heads * s.window * s.head_dim
    rc = _dev_lib().ppsyn_normal_bf16_dev(ptr, n, 0, seed, kv_stream(slot, layer, kv, s.n_layers),
                                          normal_scale(KV_SIGMA), cuda_stream)
    if rc != 0:
        raise RuntimeError("device KV fill failed: cuda error %d" % rc)
