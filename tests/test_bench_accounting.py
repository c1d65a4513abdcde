"""The bench's algorithmic bytes (the roofline numerators) against the engine's own
weight shapes (CPU).

bench.py counts the weights one tick streams with a closed formula over the model
shape.  Here the same quantity comes from the C library's weight table
(pp_weight_shape): every matrix the tick reads whole, times its bf16 size.  The
embedding tables are excluded (a tick reads 17 rows of them per slot), and so are the
fp32 RMSNorm gains (kilobytes)."""
import importlib.util
import os

import numpy as np
import pytest

import full_duplex_speech_lockstep_gb300 as pp
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STREAMED = ["wqkv", "wo", "wgu", "wdown", "wtext", "dep_inproj", "dep_wqkv", "dep_wo", "dep_wgu",
            "dep_wdown", "dep_heads"]


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", ["tiny", "small", "full"])
def test_streamed_weight_bytes_match_the_engine_weight_table(name):
    shape = synth.PRESETS[name]
    cfg = pp.make_config(shape, 1)
    total = 0
    for w in STREAMED:
        dims, f32 = pp.pp_weight_shape(cfg, pp.WEIGHT_NAMES.index(w))
        assert not f32
        total += 2 * int(np.prod(dims))
    assert _bench().weight_bytes_streamed(shape) == total


def test_full_tick_bytes_are_the_stated_workload():
    b = _bench()
    s = synth.FULL
    # ring bytes per (slot, position): K and V of every layer, bf16
    assert b.kv_bytes_per_position(s) == s.n_layers * 2 * s.d * 2
    tick = b.weight_bytes_streamed(s) + 64 * 3000 * b.kv_bytes_per_position(s) \
        + 64 * b.kv_bytes_per_position(s)
    assert round(b.weight_bytes_streamed(s) / 1e9, 3) == 13.570
    assert round(tick / 1e9, 2) == 114.27
