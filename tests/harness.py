"""Drives the CUDA path and the CPU oracle side by side on the same seeded inputs.

Used by the GPU parity tests and by ``__graft_entry__.smoke``.  It holds no arithmetic
of the tick: it schedules sessions, feeds both sides the same inputs and compares.

Teacher forcing: every tick, each open slot of the GPU engine receives the oracle's
previous column, and rows 0..8 are forced to the oracle's tokens wherever the
schedule forces them or the oracle's top-2 logit margin is at or below the token gate
(ties within rounding could go either way on either side).  Everywhere else the GPU
takes its own greedy decision, which must then equal the oracle's.
"""
import dataclasses

import numpy as np

import os

ROWS = 17
# extra engine flags for every engine the GPU tests create (e.g. 2 = PP_FLAG_NO_PDL), so the
# same suite can check the tick under another launch mode
EXTRA_FLAGS = int(os.environ.get("PP_TEST_FLAGS", "0"))
LOGIT_TOL = 2e-2        # max |gpu - oracle| <= LOGIT_TOL * std(oracle logits)
TOKEN_MARGIN = 1e-2     # tokens must agree where the oracle's top-2 margin exceeds this


def top2_margin(v):
    v = np.asarray(v, np.float32)
    i = int(np.argmax(v))
    rest = np.delete(v, i)
    return float(v[i] - rest.max())


def initial_column(shape):
    return np.array([shape.text_vocab] + [shape.audio_card] * shape.n_q, np.int32)


@dataclasses.dataclass
class Script:
    """Per-tick inputs of one session: user codes [T, 8], forced mask/tokens [T, 17]."""
    user: np.ndarray
    fmask: np.ndarray
    forced: np.ndarray

    @property
    def T(self):
        return self.user.shape[0]


@dataclasses.dataclass
class Placement:
    slot: int
    start: int          # global tick at which the session opens
    script: Script      # it runs script.T ticks, then closes
    import_pos: int = -1     # >= 0: resume at this position (ring already filled)
    check: bool = True       # False: run on the GPU only (a neighbour, not compared)


def device_view(ptr, n, dtype="<i2"):
    """A torch tensor viewing n elements of device memory at ptr (no copy): used to read
    engine memory such as a ring block back to the host."""
    import torch

    class _Mem:
        __cuda_array_interface__ = {"shape": (int(n),), "typestr": dtype,
                                    "data": (int(ptr), False), "version": 3}
    return torch.as_tensor(_Mem(), device="cuda")


def device_weights(w_host, device="cuda"):
    import torch
    out = {}
    for k, v in w_host.items():
        if v.dtype == np.uint16:
            out[k] = torch.from_numpy(v.view(np.int16)).to(device)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(device)
    return out


def run_parity(shape, B, w_host, w_dev, placements, check_logits=True, report=None,
               oracle_sessions=None, flags=0, setup=None):
    """Run the placements on a GPU engine of B slots with teacher forcing against the
    oracle; asserts column equality and the logit tolerance every tick.  Returns a dict
    of statistics.  setup(engine), if given, runs once before the first tick (e.g. to
    fill imported sessions' rings)."""
    import torch

    import full_duplex_speech_lockstep_gb300 as pp
    import oracle

    orc = oracle.Oracle(shape, w_host)
    eng = pp.Engine(shape, B, w_dev, flags=flags | EXTRA_FLAGS)
    if setup is not None:
        setup(eng)
    T_end = max(p.start + p.script.T for p in placements)
    Vt, Va, nq = shape.text_vocab, shape.audio_card, shape.n_q
    ld = Vt + nq * Va
    logits_dev = torch.empty((B, ld), dtype=torch.float32, device="cuda")
    stats = {"ticks": 0, "max_ratio": 0.0, "gpu_decided": 0, "forced_by_gate": 0}
    sess = {}
    for t in range(T_end):
        for p in placements:
            if p.start + p.script.T == t:
                eng.close(p.slot)
                del sess[p.slot]
            if p.start == t:
                if p.import_pos >= 0:
                    eng.import_session(p.slot, p.import_pos)
                else:
                    eng.open(p.slot)
                o = (oracle_sessions or {}).get(p.slot)
                if not p.check:
                    o = None
                elif o is None:
                    o = orc.new_session()
                sess[p.slot] = [p, o, initial_column(shape)]
        prev = np.tile(initial_column(shape), (B, 1))
        user = np.zeros((B, 8), np.int32)
        fmask = np.zeros((B, ROWS), np.uint8)
        forced = np.zeros((B, ROWS), np.int32)
        expect = {}
        for slot, (p, os_, pcol) in sess.items():
            i = t - p.start
            sc = p.script
            if os_ is None:     # unchecked neighbour: free-running on the GPU
                prev[slot] = pcol
                user[slot] = sc.user[i]
                fmask[slot] = sc.fmask[i]
                forced[slot] = sc.forced[i]
                continue
            col, lt, la = orc.step(os_, pcol, sc.user[i], sc.fmask[i], sc.forced[i])
            expect[slot] = (col, lt, la)
            prev[slot] = pcol
            user[slot] = sc.user[i]
            fm = sc.fmask[i].copy()
            fm[9:] = 0
            if not fm[0] and top2_margin(lt) <= TOKEN_MARGIN:
                fm[0] = 1
                stats["forced_by_gate"] += 1
            for k in range(8):
                if not fm[k + 1] and top2_margin(la[k]) <= TOKEN_MARGIN:
                    fm[k + 1] = 1
                    stats["forced_by_gate"] += 1
            stats["gpu_decided"] += int(9 - fm[:9].sum())
            fmask[slot] = fm
            forced[slot, :9] = col[:9]
            sess[slot][2] = col
        d = lambda a: torch.from_numpy(a).cuda()
        colg = eng.step(d(prev), d(user), d(fmask), d(forced), logits=logits_dev if check_logits else None)
        torch.cuda.synchronize()
        colg = colg.cpu().numpy()
        lg = logits_dev.cpu().numpy() if check_logits else None
        for slot in range(B):
            if slot in sess and slot not in expect:
                sess[slot][2] = colg[slot].copy()
                continue
            if slot not in expect:
                assert np.all(colg[slot] == -1), (t, slot, colg[slot])
                continue
            col, lt, la = expect[slot]
            assert np.array_equal(colg[slot], col), (t, slot, colg[slot], col)
            if check_logits:
                gt = lg[slot, :Vt]
                r = np.max(np.abs(gt - lt)) / np.std(lt)
                stats["max_ratio"] = max(stats["max_ratio"], float(r))
                assert r <= LOGIT_TOL, (t, slot, "text", r)
                ga = lg[slot, Vt:].reshape(nq, Va)
                for k in range(nq):
                    r = np.max(np.abs(ga[k] - la[k])) / np.std(la[k])
                    stats["max_ratio"] = max(stats["max_ratio"], float(r))
                    assert r <= LOGIT_TOL, (t, slot, "audio", k, r)
        stats["ticks"] += 1
        if report:
            report(t, stats)
    st = eng.status()
    stats["status"] = st
    eng.close_engine()
    return stats


def greedy_script(shape, T, seed, stream=100):
    """Free-running greedy session: uniform user codes, nothing forced."""
    import synth
    user = synth.uniform_i32(T * 8, seed, stream, 0, shape.audio_card).reshape(T, 8)
    return Script(user, np.zeros((T, ROWS), np.uint8), np.zeros((T, ROWS), np.int32))
