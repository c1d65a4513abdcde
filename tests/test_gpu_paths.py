"""The two contraction paths (tcgen05 tensor cores with split-bf16 activations, CUDA
cores with fp32 activations) against each other and against the oracle (GPU)."""
import numpy as np
import pytest

import synth
from harness import Placement, device_weights, greedy_script, run_parity

pytestmark = pytest.mark.gpu


def test_cuda_core_path_parity():
    """The CUDA-core contraction path passes the same oracle gate."""
    import full_duplex_speech_lockstep_gb300 as pp
    s = synth.TINY
    w = synth.make_weights_host(s, 21, alpha="random")
    st = run_parity(s, 3, w, device_weights(w),
                    [Placement(0, 0, greedy_script(s, 40, 1)), Placement(2, 5, greedy_script(s, 30, 2))],
                    flags=pp.PP_FLAG_CUDA_CORE_GEMM)
    assert st["status"] == 0


@pytest.mark.parametrize("B", [1, 9, 64])
def test_paths_agree(B):
    """One tick from the same state: both paths' logits agree to fp32-level error."""
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    s = synth.SMALL
    w = device_weights(synth.make_weights_host(s, 22, alpha="random"))
    ld = s.text_vocab + s.n_q * s.audio_card
    outs = []
    for flags in [0, pp.PP_FLAG_CUDA_CORE_GEMM]:
        e = pp.Engine(s, B, w, flags=flags)
        for b in range(B):
            e.open(b)
        prev = torch.from_numpy(np.tile(np.array([s.text_vocab] + [s.audio_card] * 16, np.int32), (B, 1))).cuda()
        user = torch.from_numpy(synth.uniform_i32(B * 8, 3, 3, 0, 2048).reshape(B, 8)).cuda()
        lg = torch.empty((B, ld), dtype=torch.float32, device="cuda")
        fm = torch.ones((B, 17), dtype=torch.uint8, device="cuda")
        fo = torch.zeros((B, 17), dtype=torch.int32, device="cuda")
        e.step(prev, user, fm, fo, logits=lg)
        torch.cuda.synchronize()
        outs.append(lg.cpu().numpy())
        assert e.status() == 0
        e.close_engine()
    a, b = outs
    scale = np.std(a)
    assert np.max(np.abs(a - b)) <= 1e-3 * scale


def test_skip_user_steps_keeps_every_column():
    """With PP_FLAG_SKIP_USER_STEPS the depformer runs steps 0..7 only: every column and
    the text and agent-row logits are bit-identical to the 16-step tick."""
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    from harness import initial_column
    s = synth.SMALL
    w = device_weights(synth.make_weights_host(s, 23, alpha="random"))
    B, T = 6, 12
    Vt, Va = s.text_vocab, s.audio_card
    ld = Vt + 16 * Va
    user = synth.uniform_i32(T * B * 8, 4, 4, 0, Va).reshape(T, B, 8)
    runs = []
    for flags in [0, pp.PP_FLAG_SKIP_USER_STEPS]:
        e = pp.Engine(s, B, w, flags=flags)
        for b in range(B):
            e.open(b)
        prev = torch.from_numpy(np.tile(initial_column(s), (B, 1))).cuda()
        lg = torch.empty((B, ld), dtype=torch.float32, device="cuda")
        cols, logits = [], []
        for t in range(T):
            col = e.step(prev, torch.from_numpy(user[t]).cuda(), logits=lg)
            torch.cuda.synchronize()
            cols.append(col.cpu().numpy().copy())
            logits.append(lg.cpu().numpy()[:, :Vt + 8 * Va].copy())
            prev = col.clone()
        assert e.status() == 0
        e.close_engine()
        runs.append((np.array(cols), np.array(logits)))
    assert np.array_equal(runs[0][0], runs[1][0])
    assert np.array_equal(runs[0][1].view(np.uint32), runs[1][1].view(np.uint32))


@pytest.mark.parametrize("B", [5, 64])
def test_batched_user_steps_match_one_at_a_time(B):
    """Depformer steps 8..15 as one batched pass (the default) against the same steps run
    one at a time (PP_FLAG_SEQUENTIAL_USER_STEPS): steps 0..7 and the temporal stack run
    the same kernels, and steps 8..15 feed nothing back (their rows are the user codes and
    the cache resets every frame), so every column and the text and agent-step logits are
    bit-identical; the user steps' logits agree to fp32 rounding (the batched
    contractions may split K differently)."""
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    from harness import initial_column
    s = synth.SMALL
    w = device_weights(synth.make_weights_host(s, 24, alpha="random"))
    T = 6
    Vt, Va = s.text_vocab, s.audio_card
    ld = Vt + 16 * Va
    user = synth.uniform_i32(T * B * 8, 5, 5, 0, Va).reshape(T, B, 8)
    runs = []
    for flags in [0, pp.PP_FLAG_SEQUENTIAL_USER_STEPS]:
        e = pp.Engine(s, B, w, flags=flags)
        for b in range(B):
            if b % 7 != 3:          # a few closed slots in between
                e.open(b)
        prev = torch.from_numpy(np.tile(initial_column(s), (B, 1))).cuda()
        lg = torch.empty((B, ld), dtype=torch.float32, device="cuda")
        cols, logits = [], []
        for t in range(T):
            col = e.step(prev, torch.from_numpy(user[t]).cuda(), logits=lg)
            torch.cuda.synchronize()
            cols.append(col.cpu().numpy().copy())
            logits.append(lg.cpu().numpy().copy())
            prev = col.clone()
        assert e.status() == 0
        runs.append((np.array(cols), np.array(logits), e.kernel_count()))
        e.close_engine()
    (ca, la, na), (cb, lb, nb) = runs
    assert na < nb                        # the batched pass launches fewer kernels
    assert np.array_equal(ca, cb)
    live = [b for b in range(B) if b % 7 != 3]
    head = Vt + 8 * Va
    assert np.array_equal(la[:, live, :head].view(np.uint32), lb[:, live, :head].view(np.uint32))
    ua, ub = la[:, live, head:], lb[:, live, head:]
    assert np.all(np.isfinite(ua))
    assert np.max(np.abs(ua - ub)) <= 1e-4 * np.std(ub)   # measured: 1.5e-5


@pytest.mark.parametrize("shape_name", ["tiny", "small"])
def test_wide_tiles_parity(shape_name):
    """256-row weight tiles (PP_FLAG_WIDE_TILES, two accumulator halves sharing each
    activation tile) pass the oracle gate; the tiny and small models give ragged tiles
    (FFN 704 and 1408 gate/up pairs over 128-pair tiles)."""
    import full_duplex_speech_lockstep_gb300 as pp
    s = synth.PRESETS[shape_name]
    w = synth.make_weights_host(s, 25, alpha="random")
    st = run_parity(s, 3, w, device_weights(w),
                    [Placement(0, 0, greedy_script(s, 24, 3)), Placement(2, 4, greedy_script(s, 16, 4))],
                    flags=pp.PP_FLAG_WIDE_TILES)
    assert st["status"] == 0


def test_fused_greedy_decisions_match_decision_kernels():
    """While no open slot samples, the tick takes its greedy decisions inside the text and
    depformer head contractions (the last CTA of each head reduces the per-CTA best keys);
    with a sampled slot open it runs the decision kernels.  The same greedy sessions (one
    with forced rows, one joining late) in an engine of each kind: bit-identical columns
    and logits, and the fused tick launches fewer kernels."""
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    from harness import initial_column
    from synth import schedules
    s = synth.SMALL
    w = device_weights(synth.make_weights_host(s, 26, alpha="random"))
    B, T = 4, 14
    Vt, Va = s.text_vocab, s.audio_card
    ld = Vt + 16 * Va
    user = synth.uniform_i32(T * B * 8, 6, 6, 0, Va).reshape(T, B, 8)
    _, fm, fo = schedules.prefill_session(s, 27, T=T, voice=3, persona=4)
    runs = []
    for sampled_neighbour in (False, True):
        e = pp.Engine(s, B, w)
        e.open(0)
        if sampled_neighbour:   # slot 3 samples: the tick needs the decision kernels
            e.open(3)
            e.set_sampling(3, text_temperature=0.8, audio_temperature=0.5, seed=9)
        prev = np.tile(initial_column(s), (B, 1))
        lg = torch.empty((B, ld), dtype=torch.float32, device="cuda")
        cols, logits = [], []
        for t in range(T):
            if t == 3:
                e.open(1)
                prev[1] = initial_column(s)   # a fresh session's first column
            FM = np.zeros((B, 17), np.uint8)
            FO = np.zeros((B, 17), np.int32)
            FM[0], FO[0] = fm[t], fo[t]
            d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
            col = e.step(d(prev), d(user[t]), d(FM), d(FO), logits=lg).cpu().numpy()
            cols.append(col[:2].copy())
            logits.append(lg.cpu().numpy()[:2].copy())
            prev = col.copy()
            prev[2] = initial_column(s)
        assert e.status() == 0
        runs.append((np.array(cols), np.array(logits), e.kernel_count()))
        e.close_engine()
    (ca, la, na), (cb, lb, nb) = runs
    assert np.array_equal(ca, cb)
    assert np.array_equal(la.view(np.uint32), lb.view(np.uint32))
    assert na == nb   # kernel_count reports the greedy tick's launches
    print("kernels per greedy tick", na)
