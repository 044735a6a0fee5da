"""Pins of the oracle's temperature-only target sampler (brb-nv/TensorRT-LLM
PR #27, "1. Temperature-only sampling runs no filter": softmax and sampling
only, no top-k / top-p / min-p filter)."""
import numpy as np
import pytest
from scipy import special, stats

import oracle


def _softmax(s):
    return special.softmax(s.astype(np.float64))


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_draws_follow_the_softmax(T):
    rng = np.random.default_rng(41)
    V, R = 8, 60_000
    row = rng.normal(0.0, 1.5, V).astype(np.float32)
    logits = np.tile(row, (R, 1))
    seed = np.arange(R, dtype=np.uint64) + np.uint64(77)
    res = oracle.sample_temperature(logits, T, seed, np.zeros(R, np.uint64))
    p = _softmax(row / np.float32(T))
    counts = np.bincount(res.tokens, minlength=V)
    assert stats.chisquare(counts, p * R).pvalue > 1e-4
    np.testing.assert_allclose(res.probs[0], p, rtol=1e-12, atol=1e-15)


def test_probabilities_are_the_draft_positions_softmax():
    # a draft position with a zero Markov head draws from softmax(base / T):
    # the sampler's probabilities for the same row must be that softmax
    rng = np.random.default_rng(42)
    V, r = 300, 4
    base = rng.normal(0.0, 3.0, V).astype(np.float32)
    U = np.zeros((V, r), np.float32)
    Wb = np.zeros((r, V), np.float32)
    pos = oracle.draft_position(base, U, Wb, 0, 5, 6, 2, 0.8)
    smp = oracle.sample_temperature(base[None, :], 0.8, np.array([5], np.uint64),
                                    np.array([6], np.uint64), position=[2])
    np.testing.assert_allclose(smp.probs[0], pos.probs, rtol=1e-13, atol=0)
    assert smp.rowstats[0, 0] == pos.M


def test_greedy_rows_take_the_lowest_argmax():
    logits = np.array([[0.0, 3.0, 1.0, 3.0], [2.0, 2.0, 2.0, 2.0],
                       [np.nan, -np.inf, 5.0, 5.0]], np.float32)
    res = oracle.sample_temperature(logits, 1.0, np.arange(3, dtype=np.uint64),
                                    np.zeros(3, np.uint64), greedy=np.ones(3))
    assert list(res.tokens) == [1, 0, 2]
    assert (res.probs[np.arange(3), res.tokens] == 1.0).all()
    assert (res.probs.sum(axis=1) == 1.0).all()


def test_noise_is_its_own_stream_and_position_dependent():
    rng = np.random.default_rng(43)
    V, R = 1000, 400
    logits = rng.normal(0.0, 0.5, (R, V)).astype(np.float32)
    seed = rng.integers(0, 2**63, R, dtype=np.uint64)
    off = np.zeros(R, np.uint64)
    a = oracle.sample_temperature(logits, 1.0, seed, off, position=np.zeros(R))
    b = oracle.sample_temperature(logits, 1.0, seed, off, position=np.ones(R))
    assert (a.tokens != b.tokens).mean() > 0.9
    # the draft stream (0) at the same counters draws differently
    U = np.zeros((V, 2), np.float32)
    Wb = np.zeros((2, V), np.float32)
    d = np.array([oracle.draft_position(logits[i], U, Wb, 0, int(seed[i]), 0, 0,
                                        1.0).token for i in range(R)])
    assert (a.tokens != d).mean() > 0.9
