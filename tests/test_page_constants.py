"""The stated constants of the pages against the generator presets and the oracle."""
import numpy as np

import oracle
import synth
from conftest import read_constants


def test_full_shape_matches_pages():
    c = read_constants()
    s = synth.FULL
    assert (s.d, s.n_layers, s.n_heads) == (c["TEMPORAL_D"], c["TEMPORAL_LAYERS"], c["TEMPORAL_HEADS"])
    assert (s.dep_d, s.dep_layers, s.dep_heads) == (c["DEPFORMER_D"], c["DEPFORMER_LAYERS"], c["DEPFORMER_HEADS"])
    assert s.window == c["WINDOW"] and s.audio_card == c["AUDIO_CARD"]
    assert s.n_q == c["DEPFORMER_STEPS"] and 1 + s.n_q == c["COLUMN_ROWS"]
    assert c["USER_ROWS_LAST"] == c["COLUMN_ROWS"] - 1
    assert c["AGENT_ROWS_LAST"] - c["AGENT_ROWS_FIRST"] + 1 == 8


def test_initial_tokens():
    c = read_constants()
    col = oracle.initial_column(synth.FULL)
    assert col[0] == c["TEXT_INITIAL_TOKEN"] == synth.FULL.text_vocab
    assert np.all(col[1:] == c["AUDIO_INITIAL_TOKEN"])


def test_silence_frames():
    from synth import schedules
    assert schedules.SILENCE_FRAMES == read_constants()["AUDIO_SILENCE_FRAME_CNT"]
