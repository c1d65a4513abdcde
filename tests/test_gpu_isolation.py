"""Batch isolation (GPU): every session's columns and logits in a batched engine are
bit-identical to the same session run alone in a one-slot engine, whichever other
sessions join, leave or recycle slots around it."""
import os

import numpy as np
import pytest

import synth
from synth import schedules
from harness import EXTRA_FLAGS, ROWS, device_weights, initial_column

pytestmark = pytest.mark.gpu


def _run(eng, B, shape, sessions, T_end, want_logits=True):
    """Free-running greedy run of `sessions` [(slot, start, user, fmask, forced)] on
    `eng`; returns per-session (columns [T,17], logits [T, ld])."""
    import torch
    ld = shape.text_vocab + shape.n_q * shape.audio_card
    logits = torch.empty((B, ld), dtype=torch.float32, device="cuda")
    out = {i: ([], []) for i in range(len(sessions))}
    prev = {}
    live = {}
    for t in range(T_end):
        for i, (slot, start, user, fm, fo) in enumerate(sessions):
            if start + user.shape[0] == t:
                eng.close(slot)
                del live[slot]
        for i, (slot, start, user, fm, fo) in enumerate(sessions):
            if start == t:
                eng.open(slot)
                live[slot] = i
                prev[i] = initial_column(shape)
        if not live:
            continue
        P = np.tile(initial_column(shape), (B, 1))
        U = np.zeros((B, 8), np.int32)
        FM = np.zeros((B, ROWS), np.uint8)
        FO = np.zeros((B, ROWS), np.int32)
        for slot, i in live.items():
            _, start, user, fm, fo = sessions[i]
            k = t - start
            P[slot], U[slot], FM[slot], FO[slot] = prev[i], user[k], fm[k], fo[k]
        d = lambda a: torch.from_numpy(a).cuda()
        col = eng.step(d(P), d(U), d(FM), d(FO), logits=logits if want_logits else None)
        col = col.cpu().numpy()
        lg = logits.cpu().numpy() if want_logits else None
        for slot, i in live.items():
            prev[i] = col[slot].copy()
            out[i][0].append(col[slot].copy())
            if want_logits:
                out[i][1].append(lg[slot].copy())
    return out


def pp_flags_two_groups():
    import full_duplex_speech_lockstep_gb300 as pp
    return pp.PP_FLAG_TWO_GROUPS


def _check_isolation(shape, B, sessions, T_end, w_dev, flags=0):
    import full_duplex_speech_lockstep_gb300 as pp
    eng = pp.Engine(shape, B, w_dev, flags=flags | EXTRA_FLAGS)
    batched = _run(eng, B, shape, sessions, T_end)
    assert eng.status() == 0
    eng.close_engine()
    for i, (slot, start, user, fm, fo) in enumerate(sessions):
        e1 = pp.Engine(shape, 1, w_dev, flags=EXTRA_FLAGS)
        alone = _run(e1, 1, shape, [(0, 0, user, fm, fo)], user.shape[0])
        e1.close_engine()
        bc, bl = np.array(batched[i][0]), np.array(batched[i][1])
        ac, al = np.array(alone[0][0]), np.array(alone[0][1])
        assert np.array_equal(bc, ac), ("columns differ", i, slot, start)
        assert np.array_equal(bl.view(np.uint32), al.view(np.uint32)), ("logits differ", i)


def test_elastic_isolation_small():
    """B=18 (two slot groups of 9, ragged operand padding) with joins, leaves and
    recycled slots."""
    s = synth.SMALL
    w = synth.make_weights_host(s, 11, alpha="random")
    sessions = schedules.elastic_schedule(s, 3, n_slots=18, T=120, initial=9, mean_gap=5,
                                          prefill=(8, 30))
    assert len(sessions) > 18
    _check_isolation(s, 18, sessions, 120, device_weights(w), flags=pp_flags_two_groups())


def test_grouping_does_not_change_bits():
    """The same sessions in a two-group engine and a one-group engine: bit-identical."""
    import full_duplex_speech_lockstep_gb300 as pp
    s = synth.TINY
    w = device_weights(synth.make_weights_host(s, 13, alpha="random"))
    sessions = []
    for i in range(20):
        user, fm, fo = schedules.prefill_session(s, 200 + i, T=15, voice=2, persona=3)
        sessions.append((i, i % 3, user, fm, fo))
    outs = []
    for flags in [0, pp.PP_FLAG_TWO_GROUPS]:
        e = pp.Engine(s, 20, w, flags=flags | EXTRA_FLAGS)
        outs.append(_run(e, 20, s, sessions, 18))
        e.close_engine()
    for i in range(len(sessions)):
        assert np.array_equal(np.array(outs[0][i][0]), np.array(outs[1][i][0]))
        assert np.array_equal(np.array(outs[0][i][1]).view(np.uint32), np.array(outs[1][i][1]).view(np.uint32))


def test_isolation_across_engine_sizes():
    """The same session in a 64-slot engine (N = 128 operand rows) next to 63 others,
    and alone (N = 16): bit-identical."""
    s = synth.TINY
    w = synth.make_weights_host(s, 12)
    sess = []
    for i in range(64):
        user, fm, fo = schedules.prefill_session(s, 100 + i, T=20, voice=3, persona=4)
        sess.append((i, i % 5, user, fm, fo))
    _check_isolation(s, 64, sess[:1] + sess[1:], 25, device_weights(w))


def test_isolation_full_shape_attention_merge_paths():
    """Full shape (2 layers), every ring full at position 3000: slots of a 64-slot engine
    against the same sessions alone.  At B=64 most (slot, head) pairs of the tensor-core
    attention are merged on chip; alone, every pair is split across CTAs and merged
    through global partials.  Columns and logits must be bit-identical."""
    import dataclasses
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    shape = dataclasses.replace(synth.FULL, n_layers=2)
    W, seed, T = shape.window, 29, 3
    w_dev = synth.make_weights_device(shape, seed)
    stream = torch.cuda.current_stream().cuda_stream

    def fill(eng, slots_src):
        for dst, src in enumerate(slots_src):
            for l in range(shape.n_layers):
                for kv in range(2):
                    synth.ring_kv_fill_device(eng.ring_block(l, dst, kv), shape, seed, src, l,
                                              kv, stream)
            eng.import_session(dst, W)
        torch.cuda.synchronize()

    def run(eng, B, slots_src):
        ld = shape.text_vocab + shape.n_q * shape.audio_card
        logits = torch.empty((B, ld), dtype=torch.float32, device="cuda")
        prev = torch.from_numpy(np.tile(initial_column(shape), (B, 1))).cuda()
        cols, lgs = [], []
        for t in range(T):
            user = np.stack([synth.uniform_i32(8, seed, 300 + t * 64 + s, 0, shape.audio_card)
                             for s in slots_src])
            col = eng.step(prev, torch.from_numpy(user).cuda(), logits=logits)
            cols.append(col.cpu().numpy().copy())
            lgs.append(logits.cpu().numpy().copy())
            prev = col.clone()
        return np.stack(cols), np.stack(lgs)

    B = 64
    eng = pp.Engine(shape, B, w_dev, flags=EXTRA_FLAGS)
    fill(eng, list(range(B)))
    bc, bl = run(eng, B, list(range(B)))
    assert eng.status() == 0
    eng.close_engine()
    del eng
    torch.cuda.empty_cache()
    for s in (0, 37, 63):
        e1 = pp.Engine(shape, 1, w_dev, flags=EXTRA_FLAGS)
        fill(e1, [s])
        ac, al = run(e1, 1, [s])
        e1.close_engine()
        assert np.array_equal(bc[:, s], ac[:, 0]), ("columns differ", s)
        assert np.array_equal(bl[:, s].view(np.uint32), al[:, 0].view(np.uint32)), ("logits", s)


@pytest.mark.parametrize("path", ["tensor", "cuda_core"])
def test_ring_append_touches_only_open_slots_at_their_position(path):
    """Each tick appends a slot's k and v to its ring at position pos mod W, for open slots
    only (on the tensor-core path this happens in the qkv contraction's epilogue, on the
    CUDA-core path in a separate kernel): a closed slot's blocks keep every byte, an open
    slot's blocks change in the row of its position and nowhere else."""
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    from harness import device_view
    s = synth.SMALL
    B, L, H, W, Dh = 4, s.n_layers, s.n_heads, s.window, s.head_dim
    flags = pp.PP_FLAG_CUDA_CORE_GEMM if path == "cuda_core" else 0
    eng = pp.Engine(s, B, device_weights(synth.make_weights_host(s, 61)), flags=flags)
    blocks = {(l, b, kv): device_view(eng.ring_block(l, b, kv), H * W * Dh).view(H, W, Dh)
              for l in range(L) for b in range(B) for kv in range(2)}
    for v in blocks.values():
        v.fill_(0x1234)
    torch.cuda.synchronize()
    user = synth.uniform_i32(6 * B * 8, 62, 0, 0, s.audio_card).reshape(6, B, 8)
    prev = torch.from_numpy(np.tile(initial_column(s), (B, 1))).cuda()
    eng.open(0)
    for t in range(6):
        if t == 2:
            eng.open(2)
            prev[2] = torch.from_numpy(initial_column(s)).cuda()   # not the closed-slot -1s
        live = [0] if t < 2 else [0, 2]
        pos = {b: eng.pos(b) for b in live}
        before = {k: v.clone() for k, v in blocks.items()}
        prev = eng.step(prev, torch.from_numpy(user[t]).cuda()).clone()
        torch.cuda.synchronize()
        for (l, b, kv), v in blocks.items():
            if b not in live:
                assert torch.equal(v, before[(l, b, kv)]), (t, l, b, kv)
                continue
            p = pos[b] % W
            rows = torch.ones(W, dtype=torch.bool, device="cuda")
            rows[p] = False
            assert torch.equal(v[:, rows], before[(l, b, kv)][:, rows]), (t, l, b, kv)
            assert (v[:, p] != before[(l, b, kv)][:, p]).any(dim=1).all(), (t, l, b, kv)
    assert eng.status() == 0
    eng.close_engine()
