"""Seeded input generator: Philox known answers, distribution, host/host determinism."""
import os

import numpy as np

import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def test_philox_known_answers():
    n = 0
    with open(os.path.join(HERE, "golden", "philox_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            v = [int(t, 16) for t in line.split()]
            out = synth.philox(v[0:4], v[4:6])
            assert [int(x) for x in out] == v[6:10]
            n += 1
    assert n == 3


def test_normal_moments_and_bf16():
    s = synth.normal_f32(1 << 20, 7, 3, 0.02)
    assert abs(float(s.mean())) < 1e-4
    assert abs(float(s.std()) - 0.02) < 2e-4
    b = synth.normal_bf16(1 << 20, 7, 3, 0.02)
    # the bf16 value is the fp32 deviate rounded to nearest-even
    f = s.view(np.uint32)
    expect = ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(b, expect)


def test_offsets_and_streams():
    a = synth.normal_bf16(1000, 1, 5, 0.02)
    b = synth.normal_bf16(400, 1, 5, 0.02, i0=600)
    assert np.array_equal(a[600:], b)
    c = synth.normal_bf16(1000, 1, 6, 0.02)
    assert not np.array_equal(a, c)


def test_uniform_range():
    u = synth.uniform_i32(100000, 3, 9, 0, 2048)
    assert u.min() == 0 and u.max() == 2047
    assert abs(u.mean() - 1023.5) < 10


def test_weight_specs_full_param_count():
    # 32 temporal layers of 202,375,168 parameters each
    specs = {n: shp for n, shp, _, _ in synth.weight_specs(synth.FULL)}
    per_layer = sum(int(np.prod(specs[n][1:])) for n in ["wqkv", "wo", "wgu", "wdown"])
    assert per_layer == 202_375_168
