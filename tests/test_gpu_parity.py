"""CUDA path against the CPU oracle, teacher-forced, tick by tick (GPU)."""
import dataclasses

import numpy as np
import pytest

import synth
from synth import schedules
from harness import Placement, Script, device_weights, greedy_script, run_parity

pytestmark = pytest.mark.gpu


def _script(arrs):
    user, fm, fo = arrs
    return Script(user, fm, fo)


def test_tiny_config_greedy_96_ticks():
    """Tiny model, B=1, 96 greedy ticks: the 64-position ring wraps at tick 64."""
    s = synth.TINY
    w = synth.make_weights_host(s, 0)
    st = run_parity(s, 1, w, device_weights(w), [Placement(0, 0, greedy_script(s, 96, 0))])
    print("parity tiny", st)
    assert st["ticks"] == 96 and st["status"] == 0
    assert st["gpu_decided"] > 500


def test_small_ragged_batch_staggered_recycled():
    """Head dims of the full model (128 / 64), ragged tiles, B=5 with staggered joins,
    a slot recycled mid-run, random RMSNorm alphas, the 80-position ring wrapping."""
    s = synth.SMALL
    w = synth.make_weights_host(s, 2, alpha="random")
    pl = [Placement(0, 0, greedy_script(s, 130, 1)),
          Placement(1, 3, greedy_script(s, 100, 2)),
          Placement(3, 10, _script(schedules.prefill_session(s, 3, T=60, voice=5, persona=20))),
          Placement(4, 17, greedy_script(s, 50, 4)),
          Placement(3, 75, greedy_script(s, 55, 5))]    # slot 3 recycled
    st = run_parity(s, 5, w, device_weights(w), pl)
    print("parity small", st)
    assert st["status"] == 0


def test_forced_prefill_and_window_one():
    """A window of one position (attention sees only the current frame) and a forced
    prefill schedule."""
    s = dataclasses.replace(synth.TINY, window=1)
    w = synth.make_weights_host(s, 4, alpha="random")
    pl = [Placement(1, 0, _script(schedules.prefill_session(s, 9, T=40, voice=4, persona=10)))]
    st = run_parity(s, 2, w, device_weights(w), pl)
    assert st["status"] == 0
