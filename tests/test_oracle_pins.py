"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- published known answers, an independent generator, closed-form
distributions, a library GEMV/softmax/argmax, or a textbook theorem -- so that
a dropped term, a wrong sign, index or operand in the oracle fails here.

All tests are CPU-only (``-m "not gpu"``)."""
import ctypes
import ctypes.util
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle
from ancestral_draft_sampling_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
P_MIN = 1e-4  # chi-square significance used by the pages' sampling tests


def _read_kat():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            w = [int(t, 16) for t in line.split()]
            rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def test_philox_known_answers():
    rows = _read_kat()
    assert len(rows) == 3
    for ctr, key, want in rows:
        got = oracle.philox4x32_10(ctr, key)
        assert [int(x) for x in got] == want


def _curand_host():
    for name in ("/usr/local/cuda/lib64/libcurand.so",
                 ctypes.util.find_library("curand")):
        if name and os.path.exists(name):
            try:
                return ctypes.CDLL(name)
            except OSError:
                pass
    return None


@pytest.mark.parametrize("seed", [0, 1234, 0x123456789ABCDEF0, 2**64 - 1])
def test_philox_matches_curand_host_generator(seed):
    """cuRAND's host-side PHILOX4_32_10 generator is an independent
    implementation; in its default ordering block i is counter (0,0,i,0)
    under key (seed lo, seed hi)."""
    lib = _curand_host()
    if lib is None:
        pytest.skip("libcurand not available")
    gen = ctypes.c_void_p()
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) != 0:
        pytest.skip("cuRAND host generator unavailable")
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        n = 4 * 257
        out = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p),
                                  ctypes.c_size_t(n)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    mine = np.concatenate([oracle.philox4x32_10([0, 0, i, 0], key)
                           for i in range(n // 4)])
    np.testing.assert_array_equal(mine, out)


def test_noise_word_counter_layout():
    """Every field of (seed, offset, position, stream, index) reaches the
    counter or key: changing any one changes the word."""
    base = oracle.noise_word(7, 9, 3, 0, 10)
    assert base != oracle.noise_word(8, 9, 3, 0, 10)
    assert base != oracle.noise_word(7 + (1 << 32), 9, 3, 0, 10)
    assert base != oracle.noise_word(7, 10, 3, 0, 10)
    assert base != oracle.noise_word(7, 9 + (1 << 32), 3, 0, 10)
    assert base != oracle.noise_word(7, 9, 4, 0, 10)
    assert base != oracle.noise_word(7, 9, 3, 1, 10)
    # four consecutive indices share one Philox block and take its 4 words
    blk = oracle.philox4x32_10([2, 3, 9, 0], [7, 0])
    assert [oracle.noise_word(7, 9, 3, 0, v) for v in range(8, 12)] == list(blk)


@pytest.mark.parametrize("seed,offset,k,stream", [
    (0, 0, 0, 0), (2**64 - 1, 2**64 - 1, 0xFFFF, 3), (2**32, 2**32 - 1, 6, 1)])
def test_noise_words_range_is_the_published_philox(seed, offset, k, stream):
    """The range form (used for long GPU comparisons) gives, for every index
    v, word v & 3 of Philox4x32-10 at counter (v >> 2, k | stream << 16,
    offset lo, offset hi) under key (seed lo, seed hi), the function the
    known answers and cuRAND pin above."""
    n = 1030  # a ragged last block
    got = oracle.noise_words(seed, offset, k, stream, n)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    c1 = k | (stream << 16)
    want = np.concatenate([
        oracle.philox4x32_10([i, c1, offset & 0xFFFFFFFF, offset >> 32], key)
        for i in range((n + 3) // 4)])[:n]
    np.testing.assert_array_equal(got, want)


def test_gumbel_cdf_and_tails():
    """g(x) for x uniform over 32-bit words follows the standard Gumbel law
    P(g <= t) = exp(-exp(-t)); g decreases in x; the upper tail behaves like
    -log(w) for tiny w."""
    rng = np.random.Generator(np.random.PCG64(5))
    xs = rng.integers(0, 2**32, size=200_000, dtype=np.uint64)
    g = np.array([oracle.gumbel(int(x)) for x in xs])
    ks = stats.kstest(g, lambda t: np.exp(-np.exp(-t)))
    assert ks.pvalue > P_MIN, ks
    # mean of the standard Gumbel is the Euler-Mascheroni constant
    assert abs(g.mean() - np.euler_gamma) < 0.02
    # monotone decreasing in the word
    grid = [0, 1, 2, 1000, 2**20, 2**31 - 1, 2**31, 2**32 - 1000, 2**32 - 1]
    vals = [oracle.gumbel(x) for x in grid]
    assert all(a > b for a, b in zip(vals, vals[1:]))
    # upper tail: w tiny => -log(-log1p(-w)) = -log(w) + O(w)
    for x in [0, 1, 17, 4095]:
        w = (x + 0.5) * 2.0**-32
        assert abs(oracle.gumbel(x) - (-np.log(w))) < 2 * w
    # lower tail: 1-w tiny => g = -log(-log(1-w)) exactly as 1-w is exact
    for x in [2**32 - 1, 2**32 - 2]:
        one_minus_w = (2**32 - x - 0.5) * 2.0**-32
        assert abs(oracle.gumbel(x) + np.log(-np.log(one_minus_w))) < 1e-12


def test_accept_uniform_grid():
    assert oracle.accept_uniform(0) == pytest.approx(0.5 * 2**-23, rel=0)
    assert oracle.accept_uniform(2**32 - 1) == pytest.approx(1 - 0.5 * 2**-23, rel=0)
    rng = np.random.Generator(np.random.PCG64(6))
    u = np.array([oracle.accept_uniform(int(x))
                  for x in rng.integers(0, 2**32, size=50_000)])
    assert stats.kstest(u, "uniform").pvalue > P_MIN


def _tiny_workload(B, K, V, r, seed, **kw):
    return wl.make_custom(B, K, V, r, seed=seed, **kw)


def _ref_logits(w, prev, k, b):
    """float32(base + U[prev] @ Wb) with a float64 library GEMV."""
    U = w.U.astype(np.float64) if w.U.dtype == np.float32 else \
        wl.bf16_bits_to_f32(w.U).astype(np.float64)
    Wb = w.Wb.astype(np.float64) if w.Wb.dtype == np.float32 else \
        wl.bf16_bits_to_f32(w.Wb).astype(np.float64)
    bias = U[prev] @ Wb
    if w.pad_row is not None and w.pad_row[b]:
        return bias.astype(np.float32)
    return (w.base_f32()[b, k].astype(np.float64) + bias).astype(np.float32)


@pytest.mark.parametrize("bdt,wdt", [(wl.F32, wl.F32), (wl.BF16, wl.BF16),
                                     (wl.F32, wl.BF16)])
def test_logits_are_base_plus_gemv(bdt, wdt):
    w = _tiny_workload(3, 4, 1000, 32, seed=11, base_dtype=bdt, w_dtype=wdt,
                       w_std=0.3, pad_rows=[2])
    out = oracle.draft_block(w.base, w.U, w.Wb, w.d0, w.seed, w.offset, w.T,
                             pad_row=w.pad_row)
    for b in range(w.B):
        prev = w.d0[b]
        for k in range(w.K):
            ref = _ref_logits(w, prev, k, b)
            # double accumulation in two different orders: equal up to one
            # float32 rounding step
            np.testing.assert_allclose(out.logits[b, k], ref, rtol=2**-23,
                                       atol=1e-30)
            prev = out.tokens[b, k]
    assert np.isfinite(out.logits[2]).all()  # NaN base ignored on padding row
    assert np.isfinite(out.probs[2]).all()


def test_proposal_is_softmax_of_scaled_logits():
    w = _tiny_workload(2, 3, 777, 16, seed=12, T=0.7, w_std=0.5)
    out = oracle.draft_block(w.base, w.U, w.Wb, w.d0, w.seed, w.offset, w.T)
    s = (out.logits / np.float32(w.T)).astype(np.float64)
    np.testing.assert_allclose(out.probs, special.softmax(s, axis=-1),
                               rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(out.probs.sum(-1), 1.0, rtol=1e-12)
    np.testing.assert_allclose(out.rowstats[..., 0], s.max(-1), rtol=0)


def test_greedy_chain_is_argmax_chain():
    w = _tiny_workload(3, 5, 513, 24, seed=13, T=0.9, w_std=0.6,
                       greedy_rows=[0, 1, 2])
    out = oracle.draft_block(w.base, w.U, w.Wb, w.d0, w.seed, w.offset, w.T,
                             greedy=w.greedy)
    for b in range(w.B):
        prev = w.d0[b]
        for k in range(w.K):
            s = _ref_logits(w, prev, k, b) / np.float32(w.T)
            d = int(np.argmax(s))  # numpy: first occurrence of the maximum
            assert out.tokens[b, k] == d
            onehot = np.zeros(w.V)
            onehot[d] = 1
            np.testing.assert_array_equal(out.probs[b, k], onehot)
            prev = d


def test_greedy_ties_take_lowest_index():
    B, K, V, r = 1, 2, 64, 8
    base = np.zeros((B, K, V), np.float32)
    base[0, 0, [5, 9, 40]] = 3.0
    base[0, 1, [7, 8]] = 1.0
    U = np.zeros((V, r), np.float32)
    Wb = np.zeros((r, V), np.float32)
    out = oracle.draft_block(base, U, Wb, [3], [1], [0], 1.0, greedy=[1])
    assert list(out.tokens[0]) == [5, 7]


def _freq_chi2(tokens, probs):
    counts = np.bincount(tokens, minlength=len(probs)).astype(np.float64)
    exp = probs * counts.sum()
    keep = exp > 5
    counts_k = np.append(counts[keep], counts[~keep].sum())
    exp_k = np.append(exp[keep], exp[~keep].sum())
    if exp_k[-1] == 0:
        counts_k, exp_k = counts_k[:-1], exp_k[:-1]
    return stats.chisquare(counts_k, exp_k).pvalue


@pytest.mark.parametrize("V,T", [(8, 1.0), (64, 1.0), (64, 0.7)])
def test_gumbel_max_frequencies_follow_softmax(V, T):
    """Position 0 drawn over many requests (distinct seeds) with identical
    logits: frequencies match softmax(l / T) (chi-square, p = 1e-4)."""
    N, r = 100_000, 4
    rng = np.random.Generator(np.random.PCG64(V))
    row = (rng.standard_normal(V) * 1.5).astype(np.float32)
    base = np.broadcast_to(row, (N, 1, V)).copy()
    U = np.zeros((V, r), np.float32)
    Wb = np.zeros((r, V), np.float32)
    seeds = np.arange(N, dtype=np.uint64) * np.uint64(2654435761) + np.uint64(99)
    out = oracle.draft_block(base, U, Wb, np.zeros(N, np.int32), seeds,
                             np.zeros(N, np.uint64), T)
    p = special.softmax((row / np.float32(T)).astype(np.float64))
    assert _freq_chi2(out.tokens[:, 0], p) > P_MIN


def test_offset_changes_the_draw_and_is_deterministic():
    w = _tiny_workload(4, 3, 300, 8, seed=14)
    a = oracle.draft_block(w.base, w.U, w.Wb, w.d0, w.seed, w.offset, w.T)
    b = oracle.draft_block(w.base, w.U, w.Wb, w.d0, w.seed, w.offset, w.T)
    c = oracle.draft_block(w.base, w.U, w.Wb, w.d0, w.seed, w.offset + 1, w.T)
    np.testing.assert_array_equal(a.tokens, b.tokens)
    assert (a.tokens != c.tokens).any()


def test_each_position_is_conditioned_on_the_drawn_token():
    """Joint (d0, d1) frequencies equal softmax(s0)[a] * softmax(s1 | a)[b]
    with a strong Markov head, so that conditioning matters (chi-square)."""
    N, V, r = 120_000, 6, 4
    rng = np.random.Generator(np.random.PCG64(21))
    base_rows = (rng.standard_normal((2, V)) * 0.5).astype(np.float32)
    U = rng.standard_normal((V, r)).astype(np.float32)
    Wb = rng.standard_normal((r, V)).astype(np.float32)
    base = np.broadcast_to(base_rows, (N, 2, V)).copy()
    d0 = np.full(N, 2, np.int32)
    seeds = np.arange(N, dtype=np.uint64) + np.uint64(5000)
    out = oracle.draft_block(base, U, Wb, d0, seeds, np.zeros(N, np.uint64), 1.0)
    U64, W64 = U.astype(np.float64), Wb.astype(np.float64)
    l0 = (base_rows[0].astype(np.float64) + U64[2] @ W64).astype(np.float32)
    p0 = special.softmax(l0.astype(np.float64))
    joint = np.zeros((V, V))
    for a in range(V):
        l1 = (base_rows[1].astype(np.float64) + U64[a] @ W64).astype(np.float32)
        joint[a] = p0[a] * special.softmax(l1.astype(np.float64))
    cells = out.tokens[:, 0] * V + out.tokens[:, 1]
    assert _freq_chi2(cells, joint.ravel()) > P_MIN
    # and the product of marginals (no conditioning) is rejected
    marg1 = joint.sum(0)
    assert _freq_chi2(cells, np.outer(p0, marg1).ravel()) < 1e-6


def test_padding_rows_draw_from_bias_alone():
    w = _tiny_workload(3, 3, 200, 8, seed=15, w_std=0.8, pad_rows=[1])
    assert np.isnan(w.base[1]).all()
    out = oracle.draft_block(w.base, w.U, w.Wb, w.d0, w.seed, w.offset, w.T,
                             pad_row=w.pad_row)
    U64, W64 = w.U.astype(np.float64), w.Wb.astype(np.float64)
    prev = w.d0[1]
    for k in range(w.K):
        np.testing.assert_allclose(out.logits[1, k],
                                   (U64[prev] @ W64).astype(np.float32),
                                   rtol=2**-23)
        assert 0 <= out.tokens[1, k] < w.V
        assert np.isfinite(out.probs[1, k]).all()
        prev = out.tokens[1, k]


def _verify_trials(N, K, V, seed):
    """Drafts drawn ancestrally by the oracle (tiny Markov head), targets
    that depend on the drafted prefix; returns tokens, q, p."""
    rng = np.random.Generator(np.random.PCG64(seed))
    r = 3
    base_rows = (rng.standard_normal((K, V)) * 0.8).astype(np.float32)
    U = rng.standard_normal((V, r)).astype(np.float32)
    Wb = rng.standard_normal((r, V)).astype(np.float32)
    base = np.broadcast_to(base_rows, (N, K, V)).copy()
    d0 = np.full(N, 1, np.int32)
    seeds = np.arange(N, dtype=np.uint64) + np.uint64(10_000 + seed)
    dr = oracle.draft_block(base, U, Wb, d0, seeds, np.zeros(N, np.uint64), 1.0)
    # target: p_k(. | previous token) = softmax(A_k + C[prev]), prefix-dependent
    A = rng.standard_normal((K + 1, V)) * 0.7
    C = rng.standard_normal((V, V)) * 0.9

    def target_row(k, prev):
        return special.softmax(A[k] + C[prev])

    prevs = np.concatenate([d0[:, None], dr.tokens], axis=1)  # [N, K+1]
    p = np.empty((N, K + 1, V), np.float32)
    for k in range(K + 1):
        for a in range(V):
            m = prevs[:, k] == a
            p[m, k] = target_row(k, a)
    return dr.tokens, dr.probs.astype(np.float32), p, seeds, target_row


def test_standard_verification_is_lossless():
    """Textbook property of rejection verification: each emitted token is
    distributed as the target given the prefix.  Checked for the first output
    token, the second given an accepted first, and the bonus token."""
    N, K, V = 150_000, 2, 4
    tokens, q, p, seeds, target_row = _verify_trials(N, K, V, seed=31)
    res = oracle.verify_standard(q, p, tokens, seeds, np.zeros(N, np.uint64))
    acc, emit = res.accepted_len, res.emitted
    assert ((acc >= 0) & (acc <= K)).all()
    # output sequence y = drafts[:acc] + [emit]
    y0 = np.where(acc >= 1, tokens[:, 0], emit)
    assert _freq_chi2(y0, target_row(0, 1)) > P_MIN
    for a in range(V):
        m = (acc >= 1) & (tokens[:, 0] == a)
        y1 = np.where(acc[m] >= 2, tokens[m, 1], emit[m])
        assert _freq_chi2(y1, target_row(1, a)) > P_MIN
    for a in range(V):
        m = (acc == 2) & (tokens[:, 1] == a)
        if m.sum() > 2000:
            assert _freq_chi2(emit[m], target_row(2, a)) > P_MIN
    # acceptance happens with probability sum_v min(p, q) at position 0
    q0 = q[:, 0]
    p0 = p[:, 0]
    want = np.minimum(q0, p0).sum(-1).mean()
    got = (acc >= 1).mean()
    assert abs(got - want) < 5 * np.sqrt(want * (1 - want) / N)


def test_verification_identical_distributions_accept_everything():
    N, K, V = 2000, 3, 5
    rng = np.random.Generator(np.random.PCG64(41))
    q = special.softmax(rng.standard_normal((N, K, V)), axis=-1).astype(np.float32)
    tokens = np.stack([[rng.choice(V, p=q[i, k] / q[i, k].sum())
                        for k in range(K)] for i in range(N)]).astype(np.int32)
    p = np.concatenate([q, q[:, -1:]], axis=1)
    res = oracle.verify_standard(q, p, tokens, np.arange(N, dtype=np.uint64),
                                 np.zeros(N, np.uint64))
    # u * q < q holds for every u < 1 (q > 0): everything is accepted
    assert (res.accepted_len == K).all()


def test_verification_zero_target_rejects():
    """A draft the target gives probability 0 is always rejected, and the
    replacement comes from the residual, never the rejected token."""
    N, K, V = 500, 1, 4
    q = np.tile(np.array([0.7, 0.1, 0.1, 0.1], np.float32), (N, K, 1))
    p = np.tile(np.array([0.0, 0.5, 0.25, 0.25], np.float32), (N, K + 1, 1))
    tokens = np.zeros((N, K), np.int32)
    res = oracle.verify_standard(q, p, tokens, np.arange(N, dtype=np.uint64),
                                 np.zeros(N, np.uint64))
    assert (res.accepted_len == 0).all()
    assert (res.emitted != 0).all()


def test_nan_and_minus_inf_never_win():
    """Reading where the pages are silent: a NaN or -inf score never wins,
    ties keep the lower index, and a row where nothing wins draws token 0."""
    V, r = 6, 4
    U = np.zeros((V, r), np.float32)
    Wb = np.zeros((r, V), np.float32)
    inf, nan = np.float32(np.inf), np.float32(np.nan)
    rows = np.array([
        [[-inf, nan, 2.0, 2.0, nan, -inf]],   # greedy: 2 (tie -> lower index)
        [[-inf] * V],                          # nothing wins -> 0
        [[nan] * V],                           # nothing wins -> 0
        [[nan, -inf, nan, -inf, nan, -inf]],   # nothing wins -> 0
    ], dtype=np.float32)
    for row, want in zip(rows, [2, 0, 0, 0]):
        out = oracle.draft_block(row[None], U, Wb, [1], [3], [0], 1.0, greedy=[1])
        assert out.tokens[0, 0] == want
        out = oracle.draft_block(row[None], U, Wb, [1], [3], [0], 1.0)
        if want == 2:
            assert out.tokens[0, 0] in (2, 3)  # sampled: one of the finite ones
        else:
            assert out.tokens[0, 0] == 0
