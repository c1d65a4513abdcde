"""Seeded per-tick input schedules of the lockstep workloads.

Each schedule returns, per session, arrays over its ticks:
    user   int32 [T, 8]   user codes (rows 9..16 of the column)
    fmask  uint8 [T, 17]  rows forced this tick (only rows 0..8 matter)
    forced int32 [T, 17]  forced tokens
The token values of the pages' SILENCE_TOKENS / SINE_TOKENS arrays are not given
anywhere, so both are seeded 8-code stand-ins; voice prompts are uniform codes and
persona text is uniform text tokens (no tokenizer or voice files exist here).
"""
import numpy as np

from . import uniform_i32

ROWS = 17
SILENCE_FRAMES = 6   # AUDIO_SILENCE_FRAME_CNT: 6 frames = 0.5 s at 12.5 Hz

# stream ids of the schedule generators
ST_SILENCE, ST_SINE, ST_VOICE, ST_PERSONA, ST_USER, ST_RUNS = 201, 202, 203, 204, 205, 206


def silence_codes(seed, card=2048):
    return uniform_i32(8, seed, ST_SILENCE, 0, card)


def sine_codes(seed, card=2048):
    return uniform_i32(8, seed, ST_SINE, 0, card)


def prefill_session(shape, seed, T=250, voice=12, persona=120, i0=0):
    """Forced persona/voice prefill then free running:
    `voice` ticks with agent rows forced to uniform voice codes, SILENCE_FRAMES ticks of
    agent silence, `persona` ticks with the text row forced to uniform text tokens (agent
    rows silent), SILENCE_FRAMES more silence ticks, then free greedy ticks up to T.
    User rows carry the SINE placeholder during prefill and uniform codes afterwards."""
    Va, Vt = shape.audio_card, shape.text_vocab
    sil, sine = silence_codes(seed, Va), sine_codes(seed, Va)
    user = uniform_i32(T * 8, seed, ST_USER, 0, Va, i0=i0 * 8).reshape(T, 8)
    fmask = np.zeros((T, ROWS), np.uint8)
    forced = np.zeros((T, ROWS), np.int32)
    pre = min(T, voice + 2 * SILENCE_FRAMES + persona)
    user[:pre] = sine
    t = 0
    vc = uniform_i32(voice * 8, seed, ST_VOICE, 0, Va).reshape(voice, 8)
    for i in range(voice):
        if t < T:
            fmask[t, 1:9], forced[t, 1:9] = 1, vc[i]
        t += 1
    for _ in range(SILENCE_FRAMES):
        if t < T:
            fmask[t, 1:9], forced[t, 1:9] = 1, sil
        t += 1
    pt = uniform_i32(persona, seed, ST_PERSONA, 0, Vt)
    for i in range(persona):
        if t < T:
            fmask[t, 0], forced[t, 0] = 1, pt[i]
            fmask[t, 1:9], forced[t, 1:9] = 1, sil
        t += 1
    for _ in range(SILENCE_FRAMES):
        if t < T:
            fmask[t, 1:9], forced[t, 1:9] = 1, sil
        t += 1
    return user, fmask, forced


def run_silence_user_codes(shape, seed, T):
    """User codes alternating uniform runs of U{12..100} frames with m in U{1..5}
    blocks of a fixed seeded 6-frame silence pattern."""
    Va = shape.audio_card
    rng = np.random.default_rng([seed, ST_RUNS])
    pattern = uniform_i32(SILENCE_FRAMES * 8, seed, ST_SILENCE + 100, 0, Va).reshape(-1, 8)
    out = np.empty((T, 8), np.int32)
    t, i0 = 0, 0
    while t < T:
        n = int(rng.integers(12, 101))
        run = uniform_i32(n * 8, seed, ST_USER, 0, Va, i0=i0).reshape(n, 8)
        i0 += n * 8
        k = min(n, T - t)
        out[t:t + k] = run[:k]
        t += k
        m = int(rng.integers(1, 6))
        for _ in range(m):
            k = min(SILENCE_FRAMES, T - t)
            out[t:t + k] = pattern[:k]
            t += k
    return out


def staggered_sessions(shape, seed, n_slots, stride, T):
    """Slot i opens at tick stride*i and runs T ticks of greedy decoding on
    run/silence user codes (nothing forced)."""
    out = []
    for i in range(n_slots):
        user = run_silence_user_codes(shape, seed * 1000 + i, T)
        out.append((i, stride * i, user, np.zeros((T, ROWS), np.uint8),
                    np.zeros((T, ROWS), np.int32)))
    return out


def elastic_schedule(shape, seed, n_slots, T, initial, mean_gap=50, prefill=(50, 200)):
    """Sessions joining and leaving: `initial` slots open at tick 0; events arrive with
    exponential gaps of mean `mean_gap` ticks; an event is a join if a slot is free and
    a fair coin says so (or nothing is open), else a leave of a random open session.
    Each session gets a forced prefill of U{prefill} ticks, its content seeded by its
    session id (not its slot).  Returns [(slot, start, user, fmask, forced)] with each
    session's arrays cut to the ticks it actually runs."""
    rng = np.random.default_rng([seed, 7])
    free = list(range(n_slots))
    open_ = {}
    sessions = []
    next_id = 0

    def join(t):
        nonlocal next_id
        slot = free.pop(int(rng.integers(0, len(free))))
        sid = next_id
        next_id += 1
        pre = int(rng.integers(prefill[0], prefill[1] + 1))
        persona = max(0, pre - 12 - 2 * SILENCE_FRAMES)
        open_[slot] = (sid, t, pre, persona)

    def leave(slot, t):
        sid, start, pre, persona = open_.pop(slot)
        n = t - start
        if n > 0:
            user, fm, fo = prefill_session(shape, seed * 100003 + sid, T=n, voice=12,
                                           persona=persona)
            sessions.append((slot, start, user, fm, fo))
        free.append(slot)

    for _ in range(min(initial, n_slots)):
        join(0)
    t = 0.0
    while True:
        t += rng.exponential(mean_gap)
        ti = int(t)
        if ti >= T:
            break
        if free and (not open_ or rng.random() < 0.5):
            join(ti)
        else:
            slots = sorted(open_)
            leave(slots[int(rng.integers(0, len(slots)))], ti)
    for slot in sorted(open_):
        leave(slot, T)
    return sorted(sessions, key=lambda s: (s[1], s[0]))
