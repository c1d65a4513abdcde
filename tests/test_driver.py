"""Session driver bookkeeping (host only, no GPU): admission and recycle, the prefill
phases, and the acoustic delay.  The delay is checked both ways:
 - the driver's model inputs follow the one-frame shift of the acoustic codebooks;
 - with a fake engine that echoes every forced row (and produces seeded tokens
   elsewhere), the aligned frames the driver returns are the aligned frames it forced,
   one tick late, and every generated frame is reassembled from the right two columns.
"""
import numpy as np
import pytest

import full_duplex_speech_lockstep_gb300 as pp
import synth

VT, VA = 1000, 2048   # text vocabulary and audio cardinality (initial tokens 1000 / 2048)


def _frames(n, seed, stream):
    return synth.uniform_i32(n * 8, seed, stream, 0, VA).reshape(n, 8)


def _fake_engine(prev, user, mask, forced, t, B):
    """A stand-in for pp_step: forced rows take the forced token, other agent rows a
    seeded token, user rows the user codes."""
    col = synth.uniform_i32(B * 17, 41, 700 + t, 0, VA).reshape(B, 17)
    col[:, 0] = synth.uniform_i32(B, 42, 700 + t, 0, VT)
    col[:, 9:] = user
    m = mask.astype(bool)
    col[:, :9][m[:, :9]] = forced[:, :9][m[:, :9]]
    return col


def test_admission_takes_the_lowest_free_slot_and_recycles():
    d = pp.Driver(3, VT, VA)
    assert [d.open() for _ in range(3)] == [0, 1, 2]
    with pytest.raises(pp.PPError):
        d.open()                                   # PP_E_BUSY
    d.close(1)
    assert d.phase(1) == pp.PP_DRV_FREE
    assert d.open() == 1
    with pytest.raises(pp.PPError):
        d.close(5)                                 # PP_E_RANGE
    d.close(0)
    with pytest.raises(pp.PPError):
        d.close(0)                                 # PP_E_NOTLIVE


def test_prefill_phases_follow_the_pages_order():
    """voice, silence, persona, silence, live (voice + 2 x silence + persona)."""
    d = pp.Driver(1, VT, VA)
    nv, ns, npers = 3, 2, 4
    slot = d.open(voice=_frames(nv, 1, 1), persona=np.arange(npers), silence=_frames(1, 1, 2)[0],
                  silence_ticks=ns)
    expect = ([pp.PP_DRV_VOICE] * nv + [pp.PP_DRV_SILENCE] * ns + [pp.PP_DRV_PERSONA] * npers +
              [pp.PP_DRV_SILENCE] * ns + [pp.PP_DRV_LIVE] * 3)
    seen = []
    for t in range(len(expect)):
        seen.append(d.phase(slot))
        u = _frames(1, 3, 10 + t)
        prev, user, mask, forced = d.prepare(u)
        d.absorb(u, _fake_engine(prev, user, mask, forced, t, 1))
    assert seen == expect


def test_user_rows_are_fed_with_the_acoustic_delay():
    d = pp.Driver(2, VT, VA)
    d.open()
    T = 6
    frames = [_frames(2, 5, 20 + t) for t in range(T)]
    for t in range(T):
        prev, user, mask, forced = d.prepare(frames[t])
        assert user[0, 0] == frames[t][0, 0]                         # semantic: this frame
        want = frames[t - 1][0, 1:] if t > 0 else np.full(7, VA)     # acoustic: one behind
        assert np.array_equal(user[0, 1:], want)
        assert np.all(user[1] == VA)                                 # slot 1 is closed
        d.absorb(frames[t], _fake_engine(prev, user, mask, forced, t, 2))


def test_forced_frames_come_back_aligned_one_tick_late():
    """Voice and silence frames forced through the delay return unchanged, and the
    persona tokens return in the text entry, each one tick after its tick."""
    B, nv, ns, npers = 2, 4, 2, 3
    d = pp.Driver(B, VT, VA)
    voice, sil, pers = _frames(nv, 7, 1), _frames(1, 7, 2)[0], np.array([5, 6, 7])
    slot = d.open(voice=voice, persona=pers, silence=sil, silence_ticks=ns)
    T = nv + 2 * ns + npers + 4
    prev_col = None
    outs, cols = [], []
    for t in range(T):
        u = _frames(B, 9, 30 + t)
        prev, user, mask, forced = d.prepare(u)
        if t == 0:   # a fresh session starts from the initial column
            assert np.array_equal(prev[slot], [VT] + [VA] * 16)
        else:
            assert np.array_equal(prev[slot], prev_col)
        col = _fake_engine(prev, user, mask, forced, t, B)
        out = d.absorb(u, col)
        prev_col = col[slot].copy()
        outs.append(out[slot].copy())
        cols.append(col[slot].copy())
    assert np.all(outs[0] == -1)                    # the first tick completes no frame
    aligned = list(voice) + [sil] * ns + [sil] * npers + [sil] * ns
    for f, fr in enumerate(aligned):                # frame f is returned by tick f+1
        assert np.array_equal(outs[f + 1][1:], fr), f
    for i, tok in enumerate(pers):
        assert outs[nv + ns + i + 1][0] == tok
    # live frames: text and codebook 0 from tick f, codebooks 1..7 from tick f+1
    for f in range(len(aligned), T - 1):
        assert outs[f + 1][0] == cols[f][0] and outs[f + 1][1] == cols[f][1]
        assert np.array_equal(outs[f + 1][2:], cols[f + 1][2:9])


def test_first_column_acoustic_rows_take_the_initial_token():
    """Tick 0 carries codebooks 1..7 of frame -1, which does not exist."""
    d = pp.Driver(1, VT, VA)
    d.open()
    prev, user, mask, forced = d.prepare(_frames(1, 11, 1))
    assert np.all(mask[0, 2:9] == 1) and np.all(forced[0, 2:9] == VA)
    assert mask[0, 0] == 0 and mask[0, 1] == 0      # text and codebook 0 are free


def test_bad_codes_are_rejected():
    d = pp.Driver(1, VT, VA)
    with pytest.raises(pp.PPError):
        d.open(voice=np.full((1, 8), VA + 1))
    with pytest.raises(pp.PPError):
        d.open(persona=np.array([VT + 1]))
    d.open()
    bad = _frames(1, 13, 1)
    bad[0, 3] = -5
    with pytest.raises(pp.PPError):
        d.prepare(bad)
