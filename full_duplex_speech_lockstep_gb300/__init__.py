"""GB300-native lockstep decode tick of the PersonaPlex / Moshi RQ-Transformer.

Thin Python binding of ``libpp.so`` (``include/pp.h``): the functions below have the C
ABI's names and only marshal arguments; every step of the tick runs in the library's
CUDA kernels.  PyTorch is used for device memory and streams only.

    import full_duplex_speech_lockstep_gb300 as pp
    eng = pp.Engine(shape, max_batch, weights)   # weights: dict of device tensors
    eng.open(0)
    col = eng.step(prev_column, user_codes)      # int32 [max_batch, 17] device tensor

There is no CPU fallback: if the library is missing or fails to load, this module
raises.
"""
import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(HERE, "libpp.so")

ROWS = 17
PP_OK, PP_EINVAL, PP_E_BUSY, PP_E_RANGE, PP_E_NOTLIVE, PP_E_CUDA, PP_E_NOSPACE = 0, -1, -2, -3, -4, -5, -6
PP_S_NAN, PP_S_INDEX, PP_S_TIMEOUT = 0x1, 0x2, 0x4
ERRORS = {PP_EINVAL: "PP_EINVAL", PP_E_BUSY: "PP_E_BUSY", PP_E_RANGE: "PP_E_RANGE",
          PP_E_NOTLIVE: "PP_E_NOTLIVE", PP_E_CUDA: "PP_E_CUDA", PP_E_NOSPACE: "PP_E_NOSPACE"}

# Order of enum pp_weight in pp.h.
WEIGHT_NAMES = ["emb_text", "emb_audio", "attn_alpha", "wqkv", "wo", "mlp_alpha", "wgu",
                "wdown", "out_alpha", "wtext", "dep_inproj", "dep_emb_text", "dep_emb_audio",
                "dep_attn_alpha", "dep_wqkv", "dep_wo", "dep_mlp_alpha", "dep_wgu",
                "dep_wdown", "dep_out_alpha", "dep_heads"]
PP_W_COUNT = len(WEIGHT_NAMES)

# Every function pp.h declares (checked against the header and the library by the tests).
EXPORTS = ["pp_weight_shape", "pp_workspace_bytes", "pp_create", "pp_destroy",
           "pp_session_open", "pp_session_close", "pp_session_import", "pp_session_pos",
           "pp_ring_block", "pp_step", "pp_step_host", "pp_status", "pp_step_kernel_count",
           "pp_profile_step", "pp_ring_attention_scratch_bytes", "pp_ring_attention",
           "pp_ring_attention_noalloc", "pp_rvq_dequantize", "pp_driver_create",
           "pp_driver_destroy", "pp_driver_open", "pp_driver_close", "pp_driver_phase",
           "pp_driver_prepare", "pp_driver_absorb", "pp_driver_tick", "pp_session_sampling",
           "pp_sample", "pp_test_faults"]

# enum pp_kernel_kind
KERNEL_KINDS = ["begin", "norm", "qkv", "rope_ring", "attn", "oproj", "gateup", "down",
                "text_head", "dep_inproj", "dep_norm", "dep_qkv", "dep_attn", "dep_oproj",
                "dep_gateup", "dep_down", "dep_head", "finish", "dep_persist"]


class PPError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__("%s failed: %s (%d)" % (fn, ERRORS.get(code, "?"), code))
        self.code = code


class pp_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ["d_model", "n_layers", "n_heads", "ffn", "text_vocab", "audio_card", "n_q",
                 "dep_d", "dep_layers", "dep_heads", "dep_ffn", "window", "max_batch"]] + [
        ("eps", ctypes.c_float), ("rope_base", ctypes.c_float), ("flags", ctypes.c_int32)]

PP_FLAG_CUDA_CORE_GEMM = 0x1
PP_FLAG_NO_PDL = 0x2
PP_FLAG_TWO_GROUPS = 0x4
PP_FLAG_SKIP_USER_STEPS = 0x8
PP_FLAG_SEQUENTIAL_USER_STEPS = 0x10
PP_FLAG_WIDE_TILES = 0x20
PP_FLAG_LOW_LATENCY = 0x40


class pp_sampling(ctypes.Structure):
    """Per-session sampling parameters (temperature <= 0 keeps a stream greedy)."""
    _fields_ = [("text_temperature", ctypes.c_float), ("text_top_k", ctypes.c_int32),
                ("text_top_p", ctypes.c_float), ("repetition_penalty", ctypes.c_float),
                ("penalty_window", ctypes.c_int32), ("audio_temperature", ctypes.c_float),
                ("audio_top_k", ctypes.c_int32), ("audio_top_p", ctypes.c_float),
                ("seed", ctypes.c_uint64)]


SAMPLE_HISTORY = 256   # the longest repetition-penalty window


class pp_weights(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p * PP_W_COUNT)]


_lib = None


def lib():
    """Load libpp.so (building it first if it is missing or older than its sources)."""
    global _lib
    if _lib is None:
        from . import build
        build.build()
        if not os.path.exists(SO):
            raise RuntimeError("libpp.so is missing; run __graft_entry__.build()")
        L = ctypes.CDLL(SO)
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.pp_weight_shape.argtypes = [P, I, P, P, P]
        L.pp_weight_shape.restype = I
        L.pp_workspace_bytes.argtypes = [P]
        L.pp_workspace_bytes.restype = ctypes.c_size_t
        L.pp_create.argtypes = [P, P, P, ctypes.c_size_t, P]
        L.pp_create.restype = I
        L.pp_destroy.argtypes = [P]
        L.pp_destroy.restype = None
        for f in ["pp_session_open", "pp_session_close"]:
            getattr(L, f).argtypes = [P, I]
            getattr(L, f).restype = I
        L.pp_session_import.argtypes = [P, I, I64]
        L.pp_session_import.restype = I
        L.pp_session_pos.argtypes = [P, I, P]
        L.pp_session_pos.restype = I
        L.pp_ring_block.argtypes = [P, I, I, I, P]
        L.pp_ring_block.restype = I
        L.pp_step.argtypes = [P] * 8
        L.pp_step.restype = I
        L.pp_step_host.argtypes = [P] * 8
        L.pp_step_host.restype = I
        L.pp_status.argtypes = [P, P, P]
        L.pp_status.restype = I
        L.pp_step_kernel_count.argtypes = [P]
        L.pp_step_kernel_count.restype = I
        L.pp_test_faults.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P]
        L.pp_test_faults.restype = I
        L.pp_profile_step.argtypes = [P] * 10
        L.pp_profile_step.restype = I
        L.pp_ring_attention_scratch_bytes.argtypes = [I, I, I, I]
        L.pp_ring_attention_scratch_bytes.restype = ctypes.c_size_t
        L.pp_ring_attention.argtypes = [P, P, P, I64, P, I, I, I, I, P, P, P, ctypes.c_size_t, P]
        L.pp_ring_attention.restype = I
        L.pp_ring_attention_noalloc.argtypes = [P, P, P, I64, P, I, I, I, I, P, P, P]
        L.pp_ring_attention_noalloc.restype = I
        L.pp_rvq_dequantize.argtypes = [P, I, I, I, P, I, I, P, P, P]
        L.pp_rvq_dequantize.restype = I
        L.pp_driver_create.argtypes = [I, I, I, ctypes.POINTER(P)]
        L.pp_driver_create.restype = I
        L.pp_driver_destroy.argtypes = [P]
        L.pp_driver_destroy.restype = None
        L.pp_driver_open.argtypes = [P, P, ctypes.POINTER(pp_prompt), ctypes.POINTER(I)]
        L.pp_driver_open.restype = I
        L.pp_driver_close.argtypes = [P, P, I]
        L.pp_driver_close.restype = I
        L.pp_driver_phase.argtypes = [P, I]
        L.pp_driver_phase.restype = I
        L.pp_driver_prepare.argtypes = [P, P, P, P, P, P]
        L.pp_driver_prepare.restype = I
        L.pp_driver_absorb.argtypes = [P, P, P, P]
        L.pp_driver_absorb.restype = I
        L.pp_driver_tick.argtypes = [P, P, P, P, P, P]
        L.pp_session_sampling.argtypes = [P, I, ctypes.POINTER(pp_sampling)]
        L.pp_session_sampling.restype = I
        F = ctypes.c_float
        L.pp_sample.argtypes = [P, I64, I, I, F, I, F, F, P, I, P, P, P, P, P]
        L.pp_sample.restype = I
        L.pp_driver_tick.restype = I
        _lib = L
    return _lib


def _check(fn, rc):
    if rc != PP_OK:
        raise PPError(fn, rc)
    return rc


def make_config(shape, max_batch, flags=0):
    """pp_config from an object with the model's dimensions (by attribute name)."""
    return pp_config(shape.d, shape.n_layers, shape.n_heads, shape.ffn, shape.text_vocab,
                     shape.audio_card, shape.n_q, shape.dep_d, shape.dep_layers,
                     shape.dep_heads, shape.dep_ffn, shape.window, int(max_batch),
                     float(shape.eps), float(shape.rope_base), int(flags))


# ---- the C ABI, one wrapper per entry point -------------------------------------------

def pp_weight_shape(cfg, which):
    dims = (ctypes.c_int64 * 4)()
    nd, f32 = ctypes.c_int(), ctypes.c_int()
    _check("pp_weight_shape", lib().pp_weight_shape(ctypes.byref(cfg), which, dims,
                                                    ctypes.byref(nd), ctypes.byref(f32)))
    return tuple(dims[:nd.value]), bool(f32.value)


def pp_workspace_bytes(cfg):
    n = lib().pp_workspace_bytes(ctypes.byref(cfg))
    if n == 0:
        raise PPError("pp_workspace_bytes", PP_EINVAL)
    return n


def pp_create(cfg, weight_ptrs, workspace_ptr, ws_bytes):
    w = pp_weights()
    for i, p in enumerate(weight_ptrs):
        w.ptr[i] = p
    h = ctypes.c_void_p()
    _check("pp_create", lib().pp_create(ctypes.byref(cfg), ctypes.byref(w), workspace_ptr,
                                        ws_bytes, ctypes.byref(h)))
    return h


def pp_destroy(h):
    lib().pp_destroy(h)


def pp_session_open(h, slot):
    return _check("pp_session_open", lib().pp_session_open(h, slot))


def pp_session_close(h, slot):
    return _check("pp_session_close", lib().pp_session_close(h, slot))


def pp_session_import(h, slot, pos):
    return _check("pp_session_import", lib().pp_session_import(h, slot, pos))


def pp_session_pos(h, slot):
    v = ctypes.c_int64()
    _check("pp_session_pos", lib().pp_session_pos(h, slot, ctypes.byref(v)))
    return v.value


def pp_ring_block(h, layer, slot, kv):
    p = ctypes.c_void_p()
    _check("pp_ring_block", lib().pp_ring_block(h, layer, slot, kv, ctypes.byref(p)))
    return p.value


def pp_step(h, prev_column, user_codes, force_mask, forced_tokens, column, logits, stream):
    return _check("pp_step", lib().pp_step(h, prev_column, user_codes, force_mask,
                                           forced_tokens, column, logits, stream))


def pp_step_host(h, prev_column, user_codes, force_mask, forced_tokens, column, logits, stream):
    return _check("pp_step_host", lib().pp_step_host(h, prev_column, user_codes, force_mask,
                                                     forced_tokens, column, logits, stream))


def pp_status(h, stream):
    v = ctypes.c_uint32()
    _check("pp_status", lib().pp_status(h, stream, ctypes.byref(v)))
    return v.value


def pp_step_kernel_count(h):
    return lib().pp_step_kernel_count(h)


PP_TEST_UMMA, PP_TEST_ATTN, PP_TEST_PERSIST = 0x1, 0x2, 0x4


def pp_test_faults(h, wait_polls, withhold, kinds, stream):
    """Failure-detection tests only: lower the bounded waits' poll budget and have
    producers of the named kernel families withhold copies (0, 0, 0 resets)."""
    return _check("pp_test_faults", lib().pp_test_faults(h, wait_polls, withhold, kinds, stream))


def pp_profile_step(h, prev_column, user_codes, force_mask, forced_tokens, column, logits,
                    stream, kind_ms, kind_launches):
    """kind_ms: ctypes double array, kind_launches: ctypes int64 array (accumulated)."""
    return _check("pp_profile_step", lib().pp_profile_step(
        h, prev_column, user_codes, force_mask, forced_tokens, column, logits, stream,
        kind_ms, kind_launches))


def pp_ring_attention_scratch_bytes(B, H, head_dim, window):
    n = lib().pp_ring_attention_scratch_bytes(B, H, head_dim, window)
    if n == 0:
        raise PPError("pp_ring_attention_scratch_bytes", PP_EINVAL)
    return n


def pp_ring_attention(q, k, v, slot_stride, n_valid, B, H, head_dim, window, out, status,
                      scratch, scratch_bytes, stream):
    return _check("pp_ring_attention", lib().pp_ring_attention(
        q, k, v, slot_stride, n_valid, B, H, head_dim, window, out, status, scratch,
        scratch_bytes, stream))


def pp_ring_attention_noalloc(q, k, v, slot_stride, n_valid, B, H, head_dim, window, out,
                              status, stream):
    """pp_ring_attention with the library's built-in scratch (no allocation)."""
    return _check("pp_ring_attention_noalloc", lib().pp_ring_attention_noalloc(
        q, k, v, slot_stride, n_valid, B, H, head_dim, window, out, status, stream))


PP_DRV_FREE, PP_DRV_VOICE, PP_DRV_SILENCE, PP_DRV_PERSONA, PP_DRV_LIVE = 0, 1, 2, 3, 4


class pp_prompt(ctypes.Structure):
    _fields_ = [("voice_frames", ctypes.c_void_p), ("n_voice", ctypes.c_int),
                ("persona_tokens", ctypes.c_void_p), ("n_persona", ctypes.c_int),
                ("silence_frame", ctypes.c_void_p), ("silence_ticks", ctypes.c_int)]


class Driver:
    """The session driver (admission, prefill, acoustic delay) over host numpy buffers.
    With an Engine, tick() runs pp_step through it; without one, prepare()/absorb() give
    the bookkeeping alone."""

    def __init__(self, max_batch, text_vocab, audio_card):
        h = ctypes.c_void_p()
        _check("pp_driver_create", lib().pp_driver_create(max_batch, text_vocab, audio_card,
                                                          ctypes.byref(h)))
        self.h, self.B = h, max_batch

    def close_driver(self):
        if self.h:
            lib().pp_driver_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close_driver()
        except Exception:
            pass

    def open(self, voice=None, persona=None, silence=None, silence_ticks=0, engine=None,
             sampling=None):
        """Admit a session (lowest free slot) and open it on `engine`; `sampling` (a
        pp_sampling) sets its sampling parameters there."""
        if sampling is not None and engine is None:
            raise ValueError("sampling parameters live on the engine: pass engine=")
        keep = []
        def arr(a):
            if a is None:
                return None, 0
            a = np.ascontiguousarray(a, dtype=np.int32)
            keep.append(a)
            return a.ctypes.data, a.shape[0]
        v, nv = arr(voice)
        p_, np_ = arr(persona)
        s_, _ = arr(silence)
        pr = pp_prompt(v, nv, p_, np_, s_, silence_ticks)
        slot = ctypes.c_int(-1)
        _check("pp_driver_open", lib().pp_driver_open(self.h, engine.h if engine else None,
                                                      ctypes.byref(pr), ctypes.byref(slot)))
        if sampling is not None:
            engine.set_sampling(slot.value, sampling)
        return slot.value

    def close(self, slot, engine=None):
        return _check("pp_driver_close",
                      lib().pp_driver_close(self.h, engine.h if engine else None, slot))

    def phase(self, slot):
        return lib().pp_driver_phase(self.h, slot)

    def prepare(self, user_frames):
        u = np.ascontiguousarray(user_frames, dtype=np.int32)
        prev = np.empty((self.B, 17), np.int32)
        user = np.empty((self.B, 8), np.int32)
        mask = np.empty((self.B, 17), np.uint8)
        forced = np.empty((self.B, 17), np.int32)
        _check("pp_driver_prepare", lib().pp_driver_prepare(
            self.h, u.ctypes.data, prev.ctypes.data, user.ctypes.data, mask.ctypes.data,
            forced.ctypes.data))
        return prev, user, mask, forced

    def absorb(self, user_frames, column):
        u = np.ascontiguousarray(user_frames, dtype=np.int32)
        c = np.ascontiguousarray(column, dtype=np.int32)
        out = np.empty((self.B, 9), np.int32)
        _check("pp_driver_absorb", lib().pp_driver_absorb(self.h, u.ctypes.data, c.ctypes.data,
                                                          out.ctypes.data))
        return out

    def tick(self, engine, user_frames):
        u = np.ascontiguousarray(user_frames, dtype=np.int32)
        out = np.empty((self.B, 9), np.int32)
        col = np.empty((self.B, 17), np.int32)
        _check("pp_driver_tick", lib().pp_driver_tick(self.h, engine.h, u.ctypes.data,
                                                      out.ctypes.data, col.ctypes.data,
                                                      engine._stream()))
        return out, col


def pp_rvq_dequantize(codes, code_stride, n_frames, n_books, codebooks, card, dim, out, status,
                      stream):
    """Latent of each frame = sum of the codebook entries its codes select (device)."""
    return _check("pp_rvq_dequantize", lib().pp_rvq_dequantize(
        codes, code_stride, n_frames, n_books, codebooks, card, dim, out, status, stream))


def pp_session_sampling(h, slot, params=None):
    """Sampling parameters of an open slot (a pp_sampling, or None for greedy)."""
    return _check("pp_session_sampling", lib().pp_session_sampling(
        h, slot, None if params is None else ctypes.byref(params)))


def pp_sample(logits, ld, rows, n, temperature, top_k, top_p, penalty, hist, hist_ld, hist_n,
              uniforms, tokens, status, stream):
    """One token per row of device logits with the caller's uniforms (device pointers)."""
    return _check("pp_sample", lib().pp_sample(logits, ld, rows, n, temperature, top_k, top_p,
                                               penalty, hist, hist_ld, hist_n, uniforms, tokens,
                                               status, stream))


def sampling(text_temperature=0.0, text_top_k=0, text_top_p=1.0, repetition_penalty=1.0,
             penalty_window=0, audio_temperature=0.0, audio_top_k=0, audio_top_p=1.0, seed=0):
    """A pp_sampling with greedy defaults."""
    return pp_sampling(text_temperature, text_top_k, text_top_p, repetition_penalty,
                       penalty_window, audio_temperature, audio_top_k, audio_top_p,
                       int(seed) & (2**64 - 1))


# ---- convenience wrapper over torch device memory ---------------------------------------

class Engine:
    """One engine over torch-owned device memory (weights dict + workspace)."""

    def __init__(self, shape, max_batch, weights, device="cuda", flags=0):
        import torch
        self.torch = torch
        self.shape = shape
        self.B = int(max_batch)
        self.cfg = make_config(shape, max_batch, flags)
        self.weights = weights
        ptrs = []
        for i, name in enumerate(WEIGHT_NAMES):
            t = weights[name]
            dims, f32 = pp_weight_shape(self.cfg, i)
            if tuple(t.shape) != dims or t.element_size() != (4 if f32 else 2):
                raise ValueError("weight %s: shape %s, expected %s" % (name, tuple(t.shape), dims))
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError("weight %s must be a contiguous CUDA tensor" % name)
            ptrs.append(t.data_ptr())
        self.ws_bytes = pp_workspace_bytes(self.cfg)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.h = pp_create(self.cfg, ptrs, self.workspace.data_ptr(), self.ws_bytes)
        self.logits_ld = shape.text_vocab + shape.n_q * shape.audio_card
        self.column = torch.empty((self.B, ROWS), dtype=torch.int32, device=device)

    def close_engine(self):
        if self.h:
            pp_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close_engine()
        except Exception:
            pass

    def _stream(self):
        return self.torch.cuda.current_stream().cuda_stream

    def open(self, slot):
        pp_session_open(self.h, slot)

    def close(self, slot):
        pp_session_close(self.h, slot)

    def set_sampling(self, slot, params=None, **kw):
        """Sampling parameters of an open slot: a pp_sampling, keyword fields of one, or
        nothing for greedy."""
        if params is None and kw:
            params = sampling(**kw)
        pp_session_sampling(self.h, slot, params)

    def import_session(self, slot, pos):
        pp_session_import(self.h, slot, pos)

    def pos(self, slot):
        return pp_session_pos(self.h, slot)

    def ring_block(self, layer, slot, kv):
        return pp_ring_block(self.h, layer, slot, kv)

    def kernel_count(self):
        return pp_step_kernel_count(self.h)

    def status(self):
        return pp_status(self.h, self._stream())

    def test_faults(self, wait_polls=0, withhold=0, kinds=0):
        pp_test_faults(self.h, wait_polls, withhold, kinds, self._stream())

    def step(self, prev_column, user_codes, force_mask=None, forced=None, logits=None,
             out=None):
        """One tick on device tensors; returns the column tensor (``out`` or the
        engine's own buffer, overwritten by the next step)."""
        col = self.column if out is None else out
        pp_step(self.h, prev_column.data_ptr(), user_codes.data_ptr(),
                None if force_mask is None else force_mask.data_ptr(),
                None if forced is None else forced.data_ptr(), col.data_ptr(),
                None if logits is None else logits.data_ptr(), self._stream())
        return col

    def profile_step(self, prev_column, user_codes, kind_ms, kind_launches, out=None):
        """One tick through the profiling graph; accumulates per-kind ms / launches."""
        col = self.column if out is None else out
        pp_profile_step(self.h, prev_column.data_ptr(), user_codes.data_ptr(), None, None,
                        col.data_ptr(), None, self._stream(), kind_ms, kind_launches)
        return col

    def step_host(self, prev_column, user_codes, force_mask, forced, column, logits=None):
        """One tick on host (numpy or pinned torch) buffers; blocks until done."""
        def ptr(a):
            if a is None:
                return None
            return a.data_ptr() if hasattr(a, "data_ptr") else a.ctypes.data
        pp_step_host(self.h, ptr(prev_column), ptr(user_codes), ptr(force_mask), ptr(forced),
                     ptr(column), ptr(logits), self._stream())
        return column
