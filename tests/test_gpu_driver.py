"""The session driver around the GPU tick (pp_driver_tick) against the oracle (GPU).

Two sessions with persona / voice prefills run through the driver on a 3-slot engine;
one is closed midway and its slot recycled for a third.  Independently of the driver,
the test restates the acoustic delay and the prefill forcing, steps the oracle with
those inputs from the GPU's previous column, and checks every column: forced rows and
user rows exactly, generated rows where the oracle's top-2 margin clears the token
gate (after the first near tie of a tick its later rows may differ legitimately, so
they are not compared).  The aligned frames the driver returns are checked against the
GPU columns they come from."""
import numpy as np
import pytest

import oracle
import synth
from harness import TOKEN_MARGIN, device_weights, initial_column, top2_margin

pytestmark = pytest.mark.gpu


class Ref:
    """Python restatement of the driver's per-session rules (delay and prefill)."""

    def __init__(self, shape, voice, persona, silence, ns):
        self.s, self.Va = shape, shape.audio_card
        self.aligned = list(voice) + [silence] * ns + [silence] * len(persona) + [silence] * ns
        self.text = [-1] * (len(voice) + ns) + list(persona) + [-1] * ns
        self.t = 0
        self.prev_user = np.full(8, self.Va, np.int32)

    def inputs(self, u):
        t = self.t
        user = np.concatenate([[u[0]], self.prev_user[1:]]).astype(np.int32)
        mask = np.zeros(17, np.uint8)
        forced = np.zeros(17, np.int32)
        if t < len(self.text) and self.text[t] >= 0:
            mask[0], forced[0] = 1, self.text[t]
        if t < len(self.aligned):
            mask[1], forced[1] = 1, self.aligned[t][0]
        if 0 < t <= len(self.aligned):
            mask[2:9], forced[2:9] = 1, self.aligned[t - 1][1:]
        elif t == 0:
            mask[2:9], forced[2:9] = 1, self.Va
        return user, mask, forced

    def advance(self, u):
        self.prev_user = np.asarray(u, np.int32).copy()
        self.t += 1


def test_driver_sessions_match_the_oracle():
    import full_duplex_speech_lockstep_gb300 as pp
    shape = synth.TINY
    w_host = synth.make_weights_host(shape, 3)
    w_dev = device_weights(w_host)
    eng = pp.Engine(shape, 3, w_dev)
    ora = oracle.Oracle(shape, w_host)
    drv = pp.Driver(3, shape.text_vocab, shape.audio_card)
    Va = shape.audio_card

    def prompt(seed):
        v = synth.uniform_i32(3 * 8, seed, 1, 0, Va).reshape(3, 8)
        p = synth.uniform_i32(4, seed, 2, 0, shape.text_vocab)
        sil = synth.uniform_i32(8, seed, 3, 0, Va)
        return v, p, sil

    sess = {}

    def admit(seed):
        v, p, sil = prompt(seed)
        slot = drv.open(voice=v, persona=p, silence=sil, silence_ticks=2, engine=eng)
        sess[slot] = {"ref": Ref(shape, v, p, sil, 2), "ora": ora.new_session(),
                      "prev": initial_column(shape), "cols": [], "outs": []}
        return slot

    assert admit(10) == 0 and admit(11) == 1
    T, close_at, checked = 24, 9, 0
    for t in range(T):
        if t == close_at:
            drv.close(0, engine=eng)
            del sess[0]
            assert admit(12) == 0                  # recycled into the freed slot
        u = synth.uniform_i32(3 * 8, 20, 100 + t, 0, Va).reshape(3, 8)
        out, col = drv.tick(eng, u)
        assert np.all(col[2] == -1) and np.all(out[2] == -1)   # slot 2 never opened
        for slot, S in sess.items():
            user, mask, forced = S["ref"].inputs(u[slot])
            co, lt, la = ora.step(S["ora"], S["prev"], user, mask, forced)
            g = col[slot]
            assert np.array_equal(g[9:], user), (t, slot)
            assert np.array_equal(g[:9][mask[:9] == 1], forced[:9][mask[:9] == 1]), (t, slot)
            margins = [top2_margin(lt)] + [top2_margin(la[k]) for k in range(8)]
            for r in range(9):                      # rows in generation order
                if mask[r]:
                    continue
                if margins[r] <= TOKEN_MARGIN:
                    break                          # a near tie: later rows may follow it
                assert g[r] == co[r], (t, slot, r, g[r], co[r])
                checked += 1
            S["prev"] = g.copy()
            S["cols"].append(g.copy())
            S["outs"].append(out[slot].copy())
            S["ref"].advance(u[slot])
    assert checked > 40
    # aligned frames: frame f = text and codebook 0 of tick f, codebooks 1..7 of tick f+1
    for S in sess.values():
        cols, outs = S["cols"], S["outs"]
        assert np.all(outs[0] == -1)
        for f in range(len(cols) - 1):
            assert outs[f + 1][0] == cols[f][0] and outs[f + 1][1] == cols[f][1]
            assert np.array_equal(outs[f + 1][2:], cols[f + 1][2:9])


def test_driver_open_sets_sampling_on_the_engine():
    """Driver.open(sampling=...) samples that session; a later admission into the same
    slot starts greedy again."""
    import full_duplex_speech_lockstep_gb300 as pp
    shape = synth.TINY
    w_host = synth.make_weights_host(shape, 3)
    eng = pp.Engine(shape, 2, device_weights(w_host))
    drv = pp.Driver(2, shape.text_vocab, shape.audio_card)
    S = pp.sampling(text_temperature=1.5, audio_temperature=1.5, seed=9)
    slot = drv.open(engine=eng, sampling=S)
    with pytest.raises(ValueError):
        drv.open(sampling=S)                       # parameters need the engine
    import torch
    lg = torch.empty((2, eng.logits_ld), dtype=torch.float32, device="cuda")
    differs = 0
    for t in range(6):
        u = synth.uniform_i32(2 * 8, 21, 200 + t, 0, shape.audio_card).reshape(2, 8)
        prev, user, mask, forced = drv.prepare(u)
        col = eng.step(torch.from_numpy(prev).cuda(), torch.from_numpy(user).cuda(),
                       torch.from_numpy(mask).cuda(), torch.from_numpy(forced).cuda(),
                       logits=lg).cpu().numpy()
        drv.absorb(u, col)
        l0 = lg[slot].cpu().numpy()
        la = l0[shape.text_vocab:].reshape(16, -1)
        differs += sum(int(col[slot, r] != oracle.argmax_f32(la[r - 1]))
                       for r in range(1, 9) if not mask[slot, r])
    assert differs > 10                            # hot sampling leaves greedy often
    drv.close(slot, engine=eng)
    assert drv.open(engine=eng) == slot            # recycled: greedy again
    u = synth.uniform_i32(2 * 8, 21, 300, 0, shape.audio_card).reshape(2, 8)
    prev, user, mask, forced = drv.prepare(u)
    col = eng.step(torch.from_numpy(prev).cuda(), torch.from_numpy(user).cuda(),
                   torch.from_numpy(mask).cuda(), torch.from_numpy(forced).cuda(),
                   logits=lg).cpu().numpy()
    l0 = lg[slot].cpu().numpy()
    assert col[slot, 0] == oracle.argmax_f32(l0[:shape.text_vocab])

