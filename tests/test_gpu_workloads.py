"""The full-shape session workloads (GPU), run at their full length:

* staggered B=8: slot i opens at tick 400*i and runs 3750 ticks (5 minutes of audio) of
  greedy decoding on run/silence user codes, so every slot's 3000-frame ring wraps; the
  whole 6550-tick schedule runs on the GPU, and at sampled ticks just after a ring has
  wrapped (and at a session's last tick) the slot's ring is copied to the host and the
  oracle steps from that exact state, teacher-forced on the GPU's tokens: logits within
  the gate, tokens equal where the oracle's top-2 margin is above the gate;
* elastic B=32: sessions join and leave on a seeded Poisson schedule (mean gap 50
  ticks) over 2000 ticks, each with a forced persona/voice prefill of 50..200 ticks;
  every session's columns and logits must be bit-identical to the same session run
  alone in a one-slot engine (logits compared through a 64-bit hash of their bits per
  tick, so that 2000 ticks of 32 x 65k logits need not be kept on the host).
"""
import os

import numpy as np
import pytest

import synth
from synth import schedules
from harness import (EXTRA_FLAGS, LOGIT_TOL, ROWS, TOKEN_MARGIN, device_view, initial_column,
                     top2_margin)

pytestmark = pytest.mark.gpu
FULL = synth.FULL
STAGGER_TICKS = int(os.environ.get("PP_STAGGER_TICKS", "3750"))
ELASTIC_TICKS = int(os.environ.get("PP_ELASTIC_TICKS", "2000"))


class _Hasher:
    """64-bit hash of each logits row's bits: sum of bits x odd multipliers, mod 2^64.
    Multiplying by an odd number is a bijection mod 2^64, so a change in any single
    entry's bits changes the hash."""

    def __init__(self, ld):
        import torch
        m = np.random.default_rng(77).integers(0, 2**62, ld, dtype=np.int64) * 2 + 1
        self.mult = torch.from_numpy(m).cuda()

    def __call__(self, lg):
        import torch
        bits = lg.view(torch.int32).to(torch.int64) & 0xFFFFFFFF
        return (bits * self.mult).sum(dim=1)


def _run_hashed(eng, B, sessions, T_end, hasher):
    """Free-running run of sessions [(slot, start, user, fmask, forced)]; returns per
    session (columns [T, 17], logit hashes [T])."""
    import torch
    ld = FULL.text_vocab + FULL.n_q * FULL.audio_card
    logits = torch.empty((B, ld), dtype=torch.float32, device="cuda")
    out = {i: ([], []) for i in range(len(sessions))}
    prev, live = {}, {}
    for t in range(T_end):
        for i, (slot, start, user, fm, fo) in enumerate(sessions):
            if start + user.shape[0] == t:
                eng.close(slot)
                del live[slot]
        for i, (slot, start, user, fm, fo) in enumerate(sessions):
            if start == t:
                eng.open(slot)
                live[slot] = i
                prev[i] = initial_column(FULL)
        if not live:
            continue
        P = np.tile(initial_column(FULL), (B, 1))
        U = np.zeros((B, 8), np.int32)
        FM = np.zeros((B, ROWS), np.uint8)
        FO = np.zeros((B, ROWS), np.int32)
        for slot, i in live.items():
            _, start, user, fm, fo = sessions[i]
            k = t - start
            P[slot], U[slot], FM[slot], FO[slot] = prev[i], user[k], fm[k], fo[k]
        d = lambda a: torch.from_numpy(a).cuda()
        col = eng.step(d(P), d(U), d(FM), d(FO), logits=logits).cpu().numpy()
        h = hasher(logits).cpu().numpy()
        for slot, i in live.items():
            prev[i] = col[slot].copy()
            out[i][0].append(col[slot].copy())
            out[i][1].append(h[slot])
    return out


def test_elastic_b32_full_shape_isolation(full_weights):
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    _, w_dev = full_weights
    B, T = 32, ELASTIC_TICKS
    sessions = schedules.elastic_schedule(FULL, 4, n_slots=B, T=T, initial=16, mean_gap=50,
                                          prefill=(50, 200))
    assert len(sessions) > 16
    hasher = _Hasher(FULL.text_vocab + FULL.n_q * FULL.audio_card)
    eng = pp.Engine(FULL, B, w_dev, flags=EXTRA_FLAGS)
    batched = _run_hashed(eng, B, sessions, T, hasher)
    assert eng.status() == 0
    eng.close_engine()
    del eng
    torch.cuda.empty_cache()
    print("elastic B=32: %d sessions over %d ticks, %d session-ticks" %
          (len(sessions), T, sum(s[2].shape[0] for s in sessions)))
    for i, (slot, start, user, fm, fo) in enumerate(sessions):
        e1 = pp.Engine(FULL, 1, w_dev, flags=EXTRA_FLAGS)
        alone = _run_hashed(e1, 1, [(0, 0, user, fm, fo)], user.shape[0], hasher)
        assert e1.status() == 0
        e1.close_engine()
        assert np.array_equal(np.array(batched[i][0]), np.array(alone[0][0])), \
            ("columns differ", i, slot, start)
        assert np.array_equal(np.array(batched[i][1]), np.array(alone[0][1])), \
            ("logits differ", i, slot, start)


def _ring_to_host(eng, slot):
    """The slot's ring, K and V, as host bf16 [L, H, W, Dh] (uint16)."""
    L, H, W, Dh = FULL.n_layers, FULL.n_heads, FULL.window, FULL.head_dim
    out = []
    for kv in range(2):
        blocks = [device_view(eng.ring_block(l, slot, kv), H * W * Dh).cpu().numpy()
                  for l in range(L)]
        out.append(np.stack(blocks).view(np.uint16).reshape(L, H, W, Dh))
    return out


def test_staggered_b8_every_ring_wraps(full_weights):
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    import oracle
    w_host, w_dev = full_weights
    B, stride, T, W = 8, 400, STAGGER_TICKS, FULL.window
    sessions = schedules.staggered_sessions(FULL, 3, n_slots=B, stride=stride, T=T)
    horizon = stride * (B - 1) + T
    Vt, Va, nq = FULL.text_vocab, FULL.audio_card, FULL.n_q
    ld = Vt + nq * Va
    # (slot, position): the first overwrite of the ring, a few ticks later, the last tick
    want = {(0, W), (0, T - 1), (3, W + 5), (7, W), (7, T - 1)} if T > W + 5 else {(0, T - 1)}
    orc = oracle.Oracle(FULL, w_host)
    eng = pp.Engine(FULL, B, w_dev, flags=EXTRA_FLAGS)
    logits = torch.empty((B, ld), dtype=torch.float32, device="cuda")
    prev = np.tile(initial_column(FULL), (B, 1))
    checked, ratios, decided = 0, [], 0
    for t in range(horizon):
        live = []
        for slot, start, user, fm, fo in sessions:
            if start + T == t:
                assert eng.pos(slot) == T            # the session ran its 3750 ticks
                eng.close(slot)
            if start == t:
                eng.open(slot)
                prev[slot] = initial_column(FULL)
            if start <= t < start + T:
                live.append(slot)
        U = np.zeros((B, 8), np.int32)
        for slot in live:
            U[slot] = sessions[slot][2][t - sessions[slot][1]]
        samples = [s for s in live if (s, t - sessions[s][1]) in want]
        states = {}
        for s in samples:
            torch.cuda.synchronize()
            rk, rv = _ring_to_host(eng, s)
            states[s] = (orc.new_session(pos=t - sessions[s][1], ring_k=rk, ring_v=rv),
                         prev[s].copy(), U[s].copy())
        d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        col = eng.step(d(prev), d(U), logits=logits if samples else None).cpu().numpy()
        if samples:
            lg = logits.cpu().numpy()
            for s in samples:
                sess, pcol, user = states[s]
                fm = np.zeros(ROWS, np.uint8)
                fm[:9] = 1                                # teacher-forced on the GPU's tokens
                fo = col[s].copy()
                ocol, lt, la = orc.step(sess, pcol, user, fm, fo)
                assert np.array_equal(col[s, 9:], user), (t, s)
                r = np.max(np.abs(lg[s, :Vt] - lt)) / np.std(lt)
                ratios.append(r)
                assert r <= LOGIT_TOL, (t, s, "text", r)
                if top2_margin(lt) > TOKEN_MARGIN:
                    assert col[s, 0] == oracle.argmax_f32(lt), (t, s, "text token")
                    decided += 1
                for k in range(nq):
                    ga = lg[s, Vt + k * Va: Vt + (k + 1) * Va]
                    r = np.max(np.abs(ga - la[k])) / np.std(la[k])
                    ratios.append(r)
                    assert r <= LOGIT_TOL, (t, s, "audio", k, r)
                    if k < 8 and top2_margin(la[k]) > TOKEN_MARGIN:
                        assert col[s, k + 1] == oracle.argmax_f32(la[k]), (t, s, "row", k + 1)
                        decided += 1
                checked += 1
        for slot in live:
            prev[slot] = col[slot]
    assert eng.status() == 0
    eng.close_engine()
    print("staggered B=8: %d ticks, %d sampled states, worst logit error %.2e x std, %d tokens "
          "decided by the GPU" % (horizon, checked, max(ratios), decided))
    assert checked == len(want)
