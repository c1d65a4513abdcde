"""Error handling on the GPU: host-detected error codes of the session table, and the
device status word (out-of-range tokens, NaN logits)."""
import numpy as np
import pytest

import synth
from harness import device_weights, initial_column

pytestmark = pytest.mark.gpu


def _engine(B=2, w=None, seed=31):
    import full_duplex_speech_lockstep_gb300 as pp
    s = synth.TINY
    if w is None:
        w = synth.make_weights_host(s, seed)
    return pp.Engine(s, B, device_weights(w)), s


def _step(eng, s, prev, user, fm=None, fo=None):
    import torch
    B = prev.shape[0]
    ld = s.text_vocab + 16 * s.audio_card
    lg = torch.empty((B, ld), dtype=torch.float32, device="cuda")
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    col = eng.step(d(prev), d(user), None if fm is None else d(fm), None if fo is None else d(fo),
                   logits=lg)
    torch.cuda.synchronize()
    return col.cpu().numpy().copy(), lg.cpu().numpy()


def test_session_table_errors():
    import full_duplex_speech_lockstep_gb300 as pp
    eng, s = _engine()
    with pytest.raises(pp.PPError) as e:
        eng.open(2)
    assert e.value.code == pp.PP_E_RANGE
    eng.open(0)
    with pytest.raises(pp.PPError) as e:
        eng.open(0)
    assert e.value.code == pp.PP_E_BUSY
    with pytest.raises(pp.PPError) as e:
        eng.close(1)
    assert e.value.code == pp.PP_E_NOTLIVE
    with pytest.raises(pp.PPError) as e:
        eng.pos(1)
    assert e.value.code == pp.PP_E_NOTLIVE
    assert eng.pos(0) == 0
    prev = np.tile(initial_column(s), (2, 1))
    _step(eng, s, prev, np.zeros((2, 8), np.int32))
    assert eng.pos(0) == 1
    eng.close(0)
    eng.open(0)
    assert eng.pos(0) == 0
    assert eng.status() == 0


def test_out_of_range_tokens_flag_and_fall_back_to_initial():
    """A previous-column token outside its table, or a forced token outside its range,
    raises PP_S_INDEX and is replaced by that row's initial token."""
    import full_duplex_speech_lockstep_gb300 as pp
    w = synth.make_weights_host(synth.TINY, 32)
    ea, s = _engine(1, w)
    eb, _ = _engine(1, w)
    ea.open(0)
    eb.open(0)
    good = initial_column(s)[None].copy()
    bad = good.copy()
    bad[0, 5] = s.audio_card + 77           # audio row out of range
    bad[0, 0] = -3                          # text row out of range
    user = np.arange(8, dtype=np.int32)[None]
    ca, la = _step(ea, s, bad, user)
    assert ea.status() & pp.PP_S_INDEX
    cb, lb = _step(eb, s, good, user)
    assert eb.status() == 0
    assert np.array_equal(ca, cb) and np.array_equal(la.view(np.uint32), lb.view(np.uint32))
    # a forced agent token out of range falls back to the initial audio token
    fm = np.zeros((1, 17), np.uint8)
    fo = np.zeros((1, 17), np.int32)
    fm[0, 3], fo[0, 3] = 1, 99999
    c2, _ = _step(ea, s, ca, user, fm, fo)
    assert c2[0, 3] == s.audio_card
    assert ea.status() & pp.PP_S_INDEX


def test_nan_logits_are_flagged_and_never_chosen():
    """A NaN row in the text head gives a NaN logit: PP_S_NAN is raised and the greedy
    token is the oracle's (which skips NaN)."""
    import full_duplex_speech_lockstep_gb300 as pp
    import oracle
    s = synth.TINY
    w = synth.make_weights_host(s, 33)
    w["wtext"] = w["wtext"].copy()
    w["wtext"][123] = 0x7FC0                 # bf16 NaN
    eng, _ = _engine(1, w)
    eng.open(0)
    prev = initial_column(s)[None]
    user = np.arange(8, dtype=np.int32)[None]
    col, lg = _step(eng, s, prev, user)
    assert eng.status() & pp.PP_S_NAN
    assert np.isnan(lg[0, 123])
    orc = oracle.Oracle(s, w)
    ocol, olt, _ = orc.step(orc.new_session(), prev[0], user[0])
    assert col[0, 0] == ocol[0] == oracle.argmax_f32(olt)
    assert col[0, 0] != 123


@pytest.mark.parametrize("shape_name,family", [("tiny", "attn"), ("small", "attn"),
                                               ("tiny", "umma"), ("small", "umma")])
def test_bounded_wait_runs_out_and_the_engine_recovers(shape_name, family):
    """A producer withholds one copy under a short poll budget (pp_test_faults): the
    consumer's bounded wait gives up, the tick still returns, and PP_S_TIMEOUT is reported.
    With the test word reset, sessions reopened in the same slots then give, tick for
    tick, bitwise the columns and logits of the same sessions in a fresh engine.  The
    tiny model's attention runs on the CUDA cores (head dim 64), the small model's on the
    tensor cores (head dim 128)."""
    import time

    import full_duplex_speech_lockstep_gb300 as pp
    s = synth.PRESETS[shape_name]
    kinds = pp.PP_TEST_ATTN if family == "attn" else pp.PP_TEST_UMMA
    wd = device_weights(synth.make_weights_host(s, 33))
    eng = pp.Engine(s, 2, wd)
    ref = pp.Engine(s, 2, wd)
    T = 5
    user = synth.uniform_i32((T + 2) * 2 * 8, 33, 9, 0, s.audio_card).reshape(T + 2, 2, 8)
    init = np.tile(initial_column(s), (2, 1))
    eng.open(0)
    eng.open(1)
    col, _ = _step(eng, s, init, user[0])
    eng.test_faults(wait_polls=4096, withhold=1, kinds=kinds)
    t0 = time.time()
    _step(eng, s, col, user[1])          # returns: the wait ran out, nothing hangs
    took = time.time() - t0
    st = eng.status()
    assert st & pp.PP_S_TIMEOUT, st
    assert st & ~(pp.PP_S_TIMEOUT | pp.PP_S_NAN) == 0, st
    assert took < 30.0, took
    eng.test_faults(0, 0, 0)
    for e in (eng, ref):
        if e is eng:
            e.close(0)
            e.close(1)
        e.open(0)
        e.open(1)
    pe, pr = init, init
    for t in range(T):
        ce, le = _step(eng, s, pe, user[t + 2])
        cr, lr = _step(ref, s, pr, user[t + 2])
        assert np.array_equal(ce, cr), t
        assert np.array_equal(le, lr), t
        pe, pr = ce, cr
    assert eng.status() == 0
    assert ref.status() == 0
