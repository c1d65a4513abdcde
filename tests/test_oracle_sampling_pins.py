"""Pins of the oracle's sampling variants to things other than itself: numpy's
independent Philox4x64-10 for the random draws, closed-form softmax probabilities for
each filter, exact tie and boundary cases for the reading's rules.

The pages pin greedy decoding; the sampling knobs they list (temperature, top-p,
repetition penalty, audio temperature) are read as the steps stated at ora_sample.
With u on a stratified grid (j + 1/2) / N, the inverse CDF returns token i for a count
of grid points within one of N * P(i), so the counts pin the sampled distribution
exactly rather than statistically.
"""
import numpy as np
import pytest
import scipy.special

import oracle


def _philox_np(counter, key):
    """numpy's Philox4x64-10 block at `counter` (numpy advances before generating)."""
    c = [int(x) for x in counter]
    carry = -1                                  # numpy adds one first: start from counter - 1
    for w in range(4):
        c[w] += carry
        carry = -1 if c[w] < 0 else 0
        c[w] %= 2**64
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64), counter=np.array(c, dtype=np.uint64))
    return bg.random_raw(4)


@pytest.mark.parametrize("counter,key", [
    ([0, 0, 0, 0], [0, 0]),
    ([7, 0, 0, 0], [0x1234, 0x5678]),
    ([2**64 - 1, 5, 9, 2**63], [2**64 - 1, 3]),
    ([123456789, 2, 0, 0], [0xDEADBEEFCAFEF00D, 0]),
])
def test_philox4x64_matches_numpy(counter, key):
    got = oracle.philox4x64(counter, key)
    assert [int(x) for x in got] == [int(x) for x in _philox_np(counter, key)]


def test_sample_uniform_is_the_counter_block_word():
    """u(seed, pos, row) = top 24 bits of word row%4 of the block (pos, row//4, 0, 0) under
    key (seed, 0), through numpy's generator; values lie on the 2^-24 grid in [0, 1)."""
    us = []
    for seed in (0, 1, 2**64 - 5):
        for pos in (0, 1, 2999, 10**9):
            for row in range(9):
                w = _philox_np([pos, row // 4, 0, 0], [seed, 0])[row % 4]
                want = float(int(w) >> 40) / 2**24
                u = oracle.sample_uniform(seed, pos, row)
                assert u == want and 0.0 <= u < 1.0
                us.append(u)
    assert len(set(us)) == len(us)             # distinct rows, positions and seeds


def _grid_counts(logits, n_draws=20000, **kw):
    toks = [oracle.sample(logits, (j + 0.5) / n_draws, **kw)[0] for j in range(n_draws)]
    return np.bincount(toks, minlength=len(logits))


def _assert_counts(counts, probs):
    n = counts.sum()
    assert np.all(np.abs(counts - n * probs) <= 1.0 + 1e-6 * n), (counts, n * probs)


def test_sample_temperature_is_the_softmax_of_scaled_logits():
    rng = np.random.default_rng(5)
    lg = rng.normal(0, 1.3, 40).astype(np.float32)
    for T in (0.3, 0.7, 1.0, 1.8):
        probs = scipy.special.softmax(lg.astype(np.float64) / T)
        _assert_counts(_grid_counts(lg, 8000, temperature=T), probs)


def test_sample_top_k_renormalises_the_k_largest():
    rng = np.random.default_rng(6)
    lg = rng.normal(0, 1.0, 60).astype(np.float32)
    for k in (1, 5, 17):
        keep = np.argsort(-lg.astype(np.float64))[:k]
        probs = np.zeros(lg.size)
        probs[keep] = scipy.special.softmax(lg[keep].astype(np.float64) / 0.8)
        _assert_counts(_grid_counts(lg, 8000, temperature=0.8, top_k=k), probs)


def test_sample_top_p_keeps_the_smallest_prefix_reaching_p():
    rng = np.random.default_rng(7)
    lg = rng.normal(0, 1.5, 50).astype(np.float32)
    p_all = scipy.special.softmax(lg.astype(np.float64) / 0.7)
    order = np.argsort(-p_all)
    for p in (0.3, 0.6, 0.9, 0.99):
        m = int(np.searchsorted(np.cumsum(p_all[order]), p) + 1)   # smallest prefix >= p
        probs = np.zeros(lg.size)
        probs[order[:m]] = p_all[order[:m]] / p_all[order[:m]].sum()
        _assert_counts(_grid_counts(lg, 8000, temperature=0.7, top_p=p), probs)


def test_sample_repetition_penalty_divides_positive_and_multiplies_negative():
    rng = np.random.default_rng(8)
    lg = rng.normal(0, 1.0, 30).astype(np.float32)
    lg[3], lg[4] = 1.7, -0.9
    hist = [3, 4, 3, 3, 11, 40, -1]            # repeats count once; out-of-range ignored
    R = 1.3
    adj = lg.astype(np.float64).copy()
    for h in {3, 4, 11}:
        adj[h] = adj[h] / R if adj[h] > 0 else adj[h] * R
    probs = scipy.special.softmax(adj)
    _assert_counts(_grid_counts(lg, 8000, penalty=R, history=hist), probs)


def test_sample_inverse_cdf_walks_the_index_order():
    # e = [1/2, 1, 1/2] (probabilities 1/4, 1/2, 1/4): index order, not size order
    lg = np.array([-np.log(2.0), 0.0, -np.log(2.0)], np.float32)
    assert oracle.sample(lg, 0.10)[0] == 0
    assert oracle.sample(lg, 0.30)[0] == 1
    assert oracle.sample(lg, 0.80)[0] == 2
    # equal logits: the first index whose running mass EXCEEDS u * Z
    eq = np.zeros(4, np.float32)
    assert [oracle.sample(eq, u)[0] for u in (0.0, 0.25, 0.5, 0.75, 0.99)] == [0, 1, 2, 3, 3]


def test_sample_limits_reduce_to_argmax():
    rng = np.random.default_rng(9)
    for trial in range(20):
        lg = rng.normal(0, 1.0, 300).astype(np.float32)
        am = oracle.argmax_f32(lg)
        for u in (0.0, 0.37, 0.999):
            assert oracle.sample(lg, u, temperature=1e-4)[0] == am
            assert oracle.sample(lg, u, top_k=1)[0] == am
            assert oracle.sample(lg, u, top_p=1e-6)[0] == am


def test_sample_ties_at_the_cuts_are_kept():
    lg = np.array([3.0, 1.0, 1.0, 0.0], np.float32)
    assert oracle.sample(lg, 0.5, top_k=2)[2] == 3           # both tokens tied at the 2nd
    eq = np.array([0.0, -1.0, -1.0, -5.0], np.float32)
    # nucleus: the run of the two equal values is kept or dropped together
    tok, amb, kept = oracle.sample(eq, 0.5, top_p=0.6)
    assert kept == 3
    assert oracle.sample(eq, 0.5, top_p=0.2)[2] == 1


def test_sample_without_finite_logits_returns_zero():
    bad = np.array([np.nan, -np.inf, np.nan], np.float32)
    assert oracle.sample(bad, 0.5) == (0, {0}, 0)
    mixed = np.array([np.nan, -np.inf, 0.5, np.inf], np.float32)
    assert oracle.sample(mixed, 0.9)[0] == 2                 # only the finite logit counts
