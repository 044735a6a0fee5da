"""Pins of the oracle's block verification (brb-nv/TensorRT-LLM PR #21,
"2. Golden sampling semantics": the block rejection_sample_method, Sun et
al. 2024; Test Coverage: lossless by chi-square).

The pages name the rule but do not state it, so these pins rest on what any
correct block verifier must satisfy:
- losslessness: the block's output, continued by plain target sampling,
  has the target's sequence distribution (chi-square over every sequence of
  a tiny vocabulary, with prefix-dependent draft and target tables).  Three
  plausible mistakes fail the same test; they are planted in a small numpy
  restatement below, which shows that the test has the power to catch them;
- with one draft it is the standard token-level rule;
- a draft equal to the target is accepted whole;
- on average it accepts at least as many drafts as the standard rule.
"""
import itertools

import numpy as np
import pytest
from scipy import stats

import oracle

V, K = 3, 2
N = 120_000


def _tables(seed):
    """Prefix-dependent conditionals: Q[prefix] (draft, prefixes shorter than
    K) and P[prefix] (target, prefixes up to K), some draft rows with a zero
    entry."""
    rng = np.random.default_rng(seed)
    P, Q = {}, {}
    for L in range(K + 1):
        for pre in itertools.product(range(V), repeat=L):
            P[pre] = rng.dirichlet(np.ones(V) * 0.8)
            if L < K:
                q = rng.dirichlet(np.ones(V) * 0.8)
                if L == 1 and pre[0] == 0:
                    q[2] = 0.0
                    q /= q.sum()
                Q[pre] = q
    return P, Q


def _draw(rng, probs):
    """One sample per row of probs [n, V] by inverse CDF."""
    c = np.cumsum(probs, axis=1)
    u = rng.random(len(probs))[:, None] * c[:, -1:]
    return np.minimum((u >= c).sum(axis=1), probs.shape[1] - 1)


def _drafts_and_rows(P, Q, rng):
    d = np.zeros((N, K), dtype=np.int32)
    q = np.zeros((N, K, V), dtype=np.float32)
    p = np.zeros((N, K + 1, V), dtype=np.float32)
    pref = [()] * N
    for k in range(K + 1):
        p[:, k] = np.array([P[pr] for pr in pref], dtype=np.float32)
        if k == K:
            break
        q[:, k] = np.array([Q[pr] for pr in pref], dtype=np.float32)
        d[:, k] = _draw(rng, q[:, k].astype(np.float64))
        pref = [pr + (int(x),) for pr, x in zip(pref, d[:, k])]
    return d, q, p


def _complete(P, d, tau, y, rng):
    """The output prefix d[:tau] + (y,), continued by target sampling to K+1
    tokens; returns the sequences as integers in base V."""
    seqs = [tuple(d[i, :tau[i]]) + (int(y[i]),) for i in range(len(d))]
    for L in range(1, K + 1):
        short = [i for i, s in enumerate(seqs) if len(s) == L]
        if not short:
            continue
        rows = np.array([P[seqs[i]] for i in short])
        nxt = _draw(rng, rows)
        for i, z in zip(short, nxt):
            seqs[i] = seqs[i] + (int(z),)
    return np.array([sum(t * V ** (K - j) for j, t in enumerate(s)) for s in seqs])


def _chi2_p(P, codes):
    expected = np.zeros(V ** (K + 1))
    for s in itertools.product(range(V), repeat=K + 1):
        pr = 1.0
        for j in range(K + 1):
            pr *= P[s[:j]][s[j]]
        expected[sum(t * V ** (K - j) for j, t in enumerate(s))] = pr
    counts = np.bincount(codes, minlength=V ** (K + 1))
    keep = expected > 0
    assert counts[~keep].sum() == 0
    e = expected[keep] * len(codes)
    return stats.chisquare(counts[keep], e * counts[keep].sum() / e.sum()).pvalue


def _restated(q, p, d, eta, g_rng, mistake=None):
    """A plain numpy restatement used only to plant mistakes (float64)."""
    n = len(d)
    w = np.ones((n, K + 1))
    for k in range(K):
        rat = p[np.arange(n), k, d[:, k]] / q[np.arange(n), k, d[:, k]]
        w[:, k + 1] = np.minimum(w[:, k] * rat, 1.0)
    tau = np.zeros(n, dtype=np.int64)
    for i in range(1, K + 1):
        if i < K:
            wi = w[:, i - 1] if mistake == "previous_weight" else w[:, i]
            r = np.maximum(wi[:, None] * p[:, i] - q[:, i], 0).sum(axis=1)
            den = r + 1 - w[:, i]
            h = np.where(den > 0, r / np.where(den > 0, den, 1), 1.0)
        else:
            h = np.ones(n) if mistake == "accept_last" else w[:, K]
        ok = eta[:, i - 1] <= h
        if mistake == "first_failure":
            tau = np.where((tau == i - 1) & ok, i, tau)
        else:
            tau = np.where(ok, i, tau)
    rows = np.zeros((n, V))
    for i in range(n):
        t = tau[i]
        if t == K:
            rows[i] = p[i, K]
        else:
            rr = np.maximum(w[i, t] * p[i, t] - q[i, t], 0)
            rows[i] = rr if rr.sum() > 0 else p[i, t]
    return tau, _draw(g_rng, rows)


@pytest.fixture(scope="module")
def sample():
    P, Q = _tables(11)
    rng = np.random.default_rng(12)
    d, q, p = _drafts_and_rows(P, Q, rng)
    seed = np.arange(N, dtype=np.uint64) + np.uint64(5000)
    off = np.zeros(N, dtype=np.uint64)
    return P, Q, d, q, p, seed, off


def test_block_verification_is_lossless(sample):
    P, Q, d, q, p, seed, off = sample
    r = oracle.verify_block(q, p, d, seed, off)
    assert ((r.accepted_len >= 0) & (r.accepted_len <= K)).all()
    codes = _complete(P, d, r.accepted_len, r.emitted, np.random.default_rng(13))
    assert _chi2_p(P, codes) > 1e-4


@pytest.mark.parametrize("mistake", ["previous_weight", "first_failure",
                                     "accept_last"])
def test_losslessness_test_catches_planted_mistakes(sample, mistake):
    P, Q, d, q, p, seed, off = sample
    rng = np.random.default_rng(14)
    eta = rng.random((N, K))
    good = _restated(q.astype(np.float64), p.astype(np.float64), d, eta,
                     np.random.default_rng(15))
    bad = _restated(q.astype(np.float64), p.astype(np.float64), d, eta,
                    np.random.default_rng(15), mistake)
    g = _complete(P, d, good[0], good[1], np.random.default_rng(16))
    b = _complete(P, d, bad[0], bad[1], np.random.default_rng(16))
    assert _chi2_p(P, g) > 1e-4
    assert _chi2_p(P, b) < 1e-6


def test_one_draft_is_the_standard_rule():
    rng = np.random.default_rng(21)
    B, V1 = 3000, 50
    q = rng.dirichlet(np.ones(V1), size=(B, 1)).astype(np.float32)
    p = rng.dirichlet(np.ones(V1), size=(B, 2)).astype(np.float32)
    d = np.array([[_draw(rng, q[i, :1].astype(np.float64))[0]] for i in range(B)],
                 dtype=np.int32)
    seed = rng.integers(0, 2**63, size=B, dtype=np.uint64)
    off = rng.integers(0, 2**40, size=B, dtype=np.uint64)
    blk = oracle.verify_block(q, p, d, seed, off)
    std = oracle.verify_standard(q, p, d, seed, off)
    # identical except where the uniform sits on the acceptance boundary
    ratio = p[np.arange(B), 0, d[:, 0]] / q[np.arange(B), 0, d[:, 0]]
    edge = np.abs(blk.eta[:, 0] - np.minimum(ratio, 1.0)) < 1e-6
    same = blk.accepted_len == std.accepted_len
    assert (same | edge).all()
    assert (blk.emitted[same] == std.emitted[same]).all()
    assert 0.2 < blk.accepted_len.mean() < 0.8


def test_draft_equal_to_target_is_accepted_whole():
    rng = np.random.default_rng(31)
    B, K2, V2 = 64, 5, 200
    q = rng.dirichlet(np.ones(V2), size=(B, K2)).astype(np.float32)
    p = np.concatenate([q, rng.dirichlet(np.ones(V2), size=(B, 1)).astype(np.float32)],
                       axis=1)
    d = rng.integers(0, V2, size=(B, K2), dtype=np.int32)
    seed = np.arange(B, dtype=np.uint64)
    off = np.full(B, 7, dtype=np.uint64)
    blk = oracle.verify_block(q, p, d, seed, off)
    std = oracle.verify_standard(q, p, d, seed, off)
    assert (blk.accepted_len == K2).all()
    np.testing.assert_array_equal(blk.emitted, std.emitted)  # the bonus row


def test_accepts_at_least_as_many_as_standard_on_average(sample):
    P, Q, d, q, p, seed, off = sample
    blk = oracle.verify_block(q, p, d, seed, off).accepted_len
    std = oracle.verify_standard(q, p, d, seed, off).accepted_len
    se = np.sqrt((blk.var() + std.var()) / N)
    assert blk.mean() >= std.mean() - 3 * se
