"""The low-latency depformer (PP_FLAG_LOW_LATENCY): all 16 codebook steps in one
persistent kernel with grid barriers (GPU).  Checked against the oracle like the default
path, for batch isolation among engines with the flag, at the full shape, and for its
bounded barrier waits."""
import numpy as np
import pytest

import synth
from synth import schedules
from harness import (EXTRA_FLAGS, Placement, Script, device_weights, greedy_script,
                     initial_column, run_parity)

pytestmark = pytest.mark.gpu


def _flag():
    import full_duplex_speech_lockstep_gb300 as pp
    return pp.PP_FLAG_LOW_LATENCY


@pytest.mark.parametrize("shape_name", ["tiny", "small"])
def test_low_latency_parity(shape_name):
    """Two sessions (one joining late, one with forced agent rows) against the oracle,
    every tick: columns exact (teacher-forced where the margin is small), all 16 steps'
    logits within the gate."""
    s = synth.PRESETS[shape_name]
    w = synth.make_weights_host(s, 41, alpha="random")
    T = 30
    user, fm, fo = schedules.prefill_session(s, 42, T=T, voice=4, persona=6)
    st = run_parity(s, 3, w, device_weights(w),
                    [Placement(0, 0, greedy_script(s, T, 5)),
                     Placement(2, 7, Script(user[:T - 7], fm[:T - 7], fo[:T - 7]))],
                    flags=_flag())
    print(shape_name, st)
    assert st["status"] == 0


def _run(eng, B, shape, sessions, T_end):
    import torch
    ld = shape.text_vocab + shape.n_q * shape.audio_card
    logits = torch.empty((B, ld), dtype=torch.float32, device="cuda")
    out = {i: ([], []) for i in range(len(sessions))}
    prev, live = {}, {}
    for t in range(T_end):
        for i, (slot, start, user, fm, fo) in enumerate(sessions):
            if start + user.shape[0] == t:
                eng.close(slot)
                del live[slot]
            if start == t:
                eng.open(slot)
                live[slot] = i
                prev[i] = initial_column(shape)
        P = np.tile(initial_column(shape), (B, 1))
        U = np.zeros((B, 8), np.int32)
        FM = np.zeros((B, 17), np.uint8)
        FO = np.zeros((B, 17), np.int32)
        for slot, i in live.items():
            _, start, user, fm, fo = sessions[i]
            k = t - start
            P[slot], U[slot], FM[slot], FO[slot] = prev[i], user[k], fm[k], fo[k]
        d = lambda a: torch.from_numpy(a).cuda()
        col = eng.step(d(P), d(U), d(FM), d(FO), logits=logits).cpu().numpy()
        lg = logits.cpu().numpy()
        for slot, i in live.items():
            prev[i] = col[slot].copy()
            out[i][0].append(col[slot].copy())
            out[i][1].append(lg[slot].copy())
    return out


def test_low_latency_isolation():
    """Sessions of a 5-slot engine with the flag, bit-identical to each session alone in a
    one-slot engine with the flag."""
    import full_duplex_speech_lockstep_gb300 as pp
    s = synth.SMALL
    wd = device_weights(synth.make_weights_host(s, 43, alpha="random"))
    sessions = []
    for i in range(6):
        user, fm, fo = schedules.prefill_session(s, 300 + i, T=12, voice=2, persona=3)
        sessions.append((i % 5, 13 * (i // 5) + i % 3, user, fm, fo))   # slot 0 recycled
    eng = pp.Engine(s, 5, wd, flags=_flag() | EXTRA_FLAGS)
    batched = _run(eng, 5, s, sessions, 27)
    assert eng.status() == 0
    eng.close_engine()
    for i, (slot, start, user, fm, fo) in enumerate(sessions):
        e1 = pp.Engine(s, 1, wd, flags=_flag() | EXTRA_FLAGS)
        alone = _run(e1, 1, s, [(0, 0, user, fm, fo)], user.shape[0])
        e1.close_engine()
        assert np.array_equal(np.array(batched[i][0]), np.array(alone[0][0])), i
        assert np.array_equal(np.array(batched[i][1]).view(np.uint32),
                              np.array(alone[0][1]).view(np.uint32)), i


def test_low_latency_full_shape_b1(full_weights):
    """The full shape at B=1: the start of the prefill workload (voice, silence, persona)
    against the oracle."""
    w_host, w_dev = full_weights
    T = 24
    user, fm, fo = schedules.prefill_session(synth.FULL, 1, T=T)
    st = run_parity(synth.FULL, 1, w_host, w_dev, [Placement(0, 0, Script(user, fm, fo))],
                    flags=_flag())
    print("full b1 low latency", st)
    assert st["status"] == 0 and st["ticks"] == T


def test_low_latency_barrier_timeout_and_recovery():
    """A CTA leaves before its first grid barrier (pp_test_faults, PP_TEST_PERSIST) under a
    short poll budget: the other CTAs' barrier waits give up, the tick returns with
    PP_S_TIMEOUT, and with the word reset, reopened sessions match a fresh engine bit for
    bit."""
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    s = synth.SMALL
    wd = device_weights(synth.make_weights_host(s, 44))
    eng = pp.Engine(s, 2, wd, flags=_flag())
    ref = pp.Engine(s, 2, wd, flags=_flag())
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    init = np.tile(initial_column(s), (2, 1))
    user = synth.uniform_i32(8 * 2 * 8, 44, 9, 0, s.audio_card).reshape(8, 2, 8)
    for e in (eng,):
        e.open(0)
        e.open(1)
    col = eng.step(d(init), d(user[0])).cpu().numpy()
    eng.test_faults(wait_polls=4096, withhold=1, kinds=pp.PP_TEST_PERSIST)
    eng.step(d(col), d(user[1]))
    torch.cuda.synchronize()
    st = eng.status()
    assert st & pp.PP_S_TIMEOUT, st
    eng.test_faults(0, 0, 0)
    eng.close(0)
    eng.close(1)
    for e in (eng, ref):
        e.open(0)
        e.open(1)
    pe, pr = init, init
    lg_e = torch.empty((2, s.text_vocab + 16 * s.audio_card), device="cuda")
    lg_r = torch.empty_like(lg_e)
    for t in range(5):
        ce = eng.step(d(pe), d(user[t + 2]), logits=lg_e).cpu().numpy()
        cr = ref.step(d(pr), d(user[t + 2]), logits=lg_r).cpu().numpy()
        assert np.array_equal(ce, cr), t
        assert torch.equal(lg_e, lg_r), t
        pe, pr = ce, cr
    assert eng.status() == 0 and ref.status() == 0
