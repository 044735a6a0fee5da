"""GPU parity of the draft-block path (through the C ABI) against the CPU
oracle, plus the properties the pages test: conditioning, chi-square of the
draws, graph replay == eager, new offset draws anew, padding rows, greedy
rows, untouched drafter logits."""
import numpy as np
import pytest
import torch
from scipy import special, stats

import ancestral_draft_sampling_gb300 as pkg
import oracle
from ancestral_draft_sampling_gb300 import workloads as wl
from tests.parity import (check_block_against_oracle, default_rows, run_draft,
                          to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _np(out):
    return tuple(t.cpu().numpy() for t in out)


# ------------------------------------------------------------------ noise
@pytest.mark.parametrize("seed,offset,k,stream", [
    (0, 0, 0, 0), (1234, 0, 3, 0), (2**64 - 1, 2**40 + 7, 6, 0),
    (99, 5, 2, 1), (99, 5, 7, 2)])
def test_noise_words_bit_exact(seed, offset, k, stream):
    n = 4099
    words, g = pkg.noise_words(seed, offset, k, stream, n)
    words = words.cpu().numpy().view(np.uint32)
    ref = np.array([oracle.noise_word(seed, offset, k, stream, v)
                    for v in range(n)], dtype=np.uint32)
    np.testing.assert_array_equal(words, ref)
    g = g.cpu().numpy()
    gref = np.array([oracle.gumbel(int(x)) for x in ref])
    # float32 log1pf/logf: a few ulp of |g| (|g| < 23)
    np.testing.assert_allclose(g, gref, rtol=0, atol=4 * 2.0**-19)


def test_gumbel_tails_bit_for_word():
    """The words at both ends of the range give the extreme Gumbel values."""
    # find words near 0 and near 2^32 among a long stream
    n = 1 << 20
    words, g = pkg.noise_words(77, 0, 0, 0, n)
    words = words.cpu().numpy().view(np.uint32)
    g = g.cpu().numpy()
    for i in [int(np.argmin(words)), int(np.argmax(words))]:
        assert abs(g[i] - oracle.gumbel(int(words[i]))) <= 4 * 2.0**-19


@pytest.mark.parametrize("seed,offset,k,stream", [
    (0, 0, 0, 0), (2**64 - 1, 2**64 - 1, 0xFFFF, 3), (2**32 - 1, 2**32, 6, 0),
    (2**32, 2**32 - 1, 3, 1), (0x9E3779B97F4A7C15, 12345, 1, 2)])
def test_folded_noise_words_bit_exact_over_a_million_counters(seed, offset, k,
                                                              stream):
    """The folded Philox the position, verification and sampler kernels run
    (rounds 1-2 folded into per-request constants) gives the published
    Philox4x32-10 words bit for bit: 2^20 words (262,144 counters) per
    (seed, offset, position, stream), 1.3 M counters over the five cases,
    with the extremes of seed, offset and the counter's position word."""
    n = 1 << 20
    words, g = pkg.noise_words(seed, offset, k, stream, n, folded=True)
    words = words.cpu().numpy().view(np.uint32)
    ref = oracle.noise_words(seed, offset, k, stream, n)
    np.testing.assert_array_equal(words, ref)
    plain, gp = pkg.noise_words(seed, offset, k, stream, n)
    np.testing.assert_array_equal(plain.cpu().numpy().view(np.uint32), ref)
    np.testing.assert_array_equal(g.cpu().numpy(), gp.cpu().numpy())


# ------------------------------------------------------- small-shape parity
SMALL_CASES = [
    # B, K, V, r, base dtype, w dtype, T, extra
    (1, 3, 4096, 64, wl.F32, wl.F32, 1.0, {}),
    (3, 4, 4100, 32, wl.BF16, wl.BF16, 0.7, {}),          # ragged V (not /8)
    (2, 2, 4099, 16, wl.F32, wl.BF16, 1.3, {}),           # odd V: scalar path
    (5, 3, 1000, 48, wl.BF16, wl.F32, 1.0, {"greedy_rows": [1, 3]}),
    (4, 3, 3000, 64, wl.F32, wl.BF16, 1.0, {"pad_rows": [0, 3]}),
    (70, 2, 2048, 32, wl.BF16, wl.F32, 1.0, {"n_spikes": 4}),   # two CTA groups
    (2, 3, 1536, 64, wl.F32, wl.F32, 0.05, {}),           # extreme T
    (2, 3, 1536, 64, wl.F32, wl.F32, 20.0, {}),
    (1, 1, 1, 16, wl.F32, wl.F32, 1.0, {}),               # V = 1
    (2, 20, 777, 32, wl.BF16, wl.F32, 0.9, {}),           # a long chain
    (1024, 1, 64, 16, wl.F32, wl.F32, 1.0, {}),           # the largest batch
    (3, 2, 130, 256, wl.BF16, wl.BF16, 1.0, {}),          # r = 256, V < 2 tiles
    # shapes the tensor-core kernel takes (bf16 head, r % 16 == 0, V % 8 == 0)
    (4, 2, 1024, 16, wl.F32, wl.BF16, 1.0, {}),           # r = 16: one K step
    (3, 2, 8, 64, wl.F32, wl.BF16, 1.0, {"greedy_rows": [0]}),  # V = 8: one part tile
    (9, 3, 2048, 32, wl.BF16, wl.BF16, 0.8, {"greedy_rows": [2]}),
    (7, 2, 4096, 48, wl.F32, wl.BF16, 1.0, {"pad_rows": [6]}),
    (20, 2, 3000, 80, wl.F32, wl.BF16, 1.3, {}),          # a whole and a part chunk
    (12, 2, 2048, 208, wl.BF16, wl.BF16, 1.0, {"n_spikes": 4}),
    (16, 3, 4096, 64, wl.F32, wl.BF16, 1.0, {}),
    (5, 2, 1000, 128, wl.BF16, wl.BF16, 0.7, {"greedy_rows": [1]}),  # ragged tile
    (33, 2, 2056, 256, wl.F32, wl.BF16, 1.0, {"pad_rows": [0, 32]}),
    (96, 2, 1024, 64, wl.BF16, wl.BF16, 1.0, {}),         # its largest batch
    (95, 1, 8192, 192, wl.F32, wl.BF16, 1.3, {}),
    (3, 64, 520, 64, wl.F32, wl.BF16, 1.0, {"greedy_rows": [1]}),  # K = 64
    # more than 96 requests: groups of at most 96, one chain each
    (128, 2, 1024, 64, wl.BF16, wl.BF16, 1.0, {}),        # 2 groups of 64
    (300, 2, 512, 64, wl.F32, wl.BF16, 1.0, {"pad_rows": [299], "greedy_rows": [97]}),
    (1024, 2, 256, 64, wl.BF16, wl.BF16, 0.9, {}),        # 11 groups
    (1, 3, 200064, 256, wl.BF16, wl.BF16, 1.0, {"n_spikes": 32}),
    # bf16 drafter logits: with r = 256, B > 64 gets one staging tile (two
    # would leave the Wb ring fewer than four stages), B <= 64 two
    (88, 2, 4096, 256, wl.BF16, wl.BF16, 1.0, {"greedy_rows": [5], "pad_rows": [87]}),
    (96, 3, 2056, 128, wl.BF16, wl.BF16, 0.8, {}),
    (48, 2, 3072, 256, wl.BF16, wl.BF16, 1.0, {"n_spikes": 4}),
]


def tc_eligible(case):
    """Shapes the tensor-core kernel takes (bf16 head, r a multiple of 16 up
    to 256, V % 8 == 0; more than 96 requests run as request groups)."""
    B, K, V, r, bdt, wdt = case[:6]
    return wdt == wl.BF16 and r % 16 == 0 and r <= 256 and V % 8 == 0


@pytest.mark.parametrize("case", SMALL_CASES, ids=lambda c: f"B{c[0]}K{c[1]}V{c[2]}r{c[3]}")
def test_small_parity(case):
    B, K, V, r, bdt, wdt, T, extra = case
    w = wl.make_custom(B, K, V, r, seed=100 + V + B, base_dtype=bdt,
                       w_dtype=wdt, T=T, w_std=0.2, **extra)
    base_before = w.base.copy()
    dev = to_device(w)
    tokens, logits, probs = _np(run_draft(w, dev))
    stats_ = check_block_against_oracle(w, tokens, logits, probs)
    assert stats_["near_tie_token_diffs"] <= 1
    # the drafter's logits are left as they are
    after = dev["base"].cpu()
    if w.base.dtype == np.uint16:
        after = after.view(torch.int16).numpy().view(np.uint16)
    else:
        after = after.numpy()
    np.testing.assert_array_equal(after, base_before)


@pytest.mark.parametrize("case", [c for c in SMALL_CASES if tc_eligible(c)],
                         ids=lambda c: f"B{c[0]}K{c[1]}V{c[2]}r{c[3]}")
def test_ffma_kernel_parity_on_tensor_core_shapes(case, monkeypatch):
    """The FFMA position kernel, forced on shapes the tensor-core kernel
    normally takes, meets the same bar."""
    monkeypatch.setenv("DSPARK_POSITION_KERNEL", "generic")
    B, K, V, r, bdt, wdt, T, extra = case
    w = wl.make_custom(B, K, V, r, seed=200 + V + B, base_dtype=bdt,
                       w_dtype=wdt, T=T, w_std=0.2, **extra)
    tokens, logits, probs = _np(run_draft(w))
    st = check_block_against_oracle(w, tokens, logits, probs,
                                    rows=default_rows(B, K, max_rows=64))
    assert st["near_tie_token_diffs"] <= 1


@pytest.mark.parametrize("case", [c for c in SMALL_CASES if tc_eligible(c)],
                         ids=lambda c: f"B{c[0]}K{c[1]}V{c[2]}r{c[3]}")
def test_tensor_core_kernel_takes_the_eligible_shapes(case, monkeypatch):
    """The shapes the parity tests count as tensor-core shapes do run the
    tensor-core kernel: forcing it succeeds and gives the default call's
    outputs bit for bit."""
    B, K, V, r, bdt, wdt, T, extra = case
    w = wl.make_custom(B, K, V, r, seed=300 + V + B, base_dtype=bdt,
                       w_dtype=wdt, T=T, w_std=0.2, **extra)
    dev = to_device(w)
    default = _np(run_draft(w, dev))
    monkeypatch.setenv("DSPARK_POSITION_KERNEL", "tc")
    forced = _np(run_draft(w, dev))
    for a, b in zip(default, forced):
        np.testing.assert_array_equal(a, b)


def test_forcing_tensor_core_kernel_on_unsupported_shape_fails(monkeypatch):
    monkeypatch.setenv("DSPARK_POSITION_KERNEL", "tc")
    w = wl.make_custom(2, 2, 1001, 64, seed=5, w_dtype=wl.BF16)
    with pytest.raises(pkg.DsparkError):
        run_draft(w)


def test_config_small_parity():
    w = wl.make_config(1)
    tokens, logits, probs = _np(run_draft(w))
    st = check_block_against_oracle(w, tokens, logits, probs)
    assert st["near_tie_token_diffs"] == 0
    ref = oracle.draft_block(w.base, w.U, w.Wb, w.d0, w.seed, w.offset, w.T)
    np.testing.assert_array_equal(tokens, ref.tokens)


def test_greedy_ties_lowest_index():
    B, K, V, r = 2, 2, 640, 16
    w = wl.make_custom(B, K, V, r, seed=3, w_std=0.0, greedy_rows=[0, 1])
    w.base[:] = 0.0
    w.base[0, 0, [300, 17, 600]] = 5.0
    w.base[1, :, :] = 1.0  # all equal -> index 0
    tokens, logits, probs = _np(run_draft(w))
    assert tokens[0, 0] == 17
    assert (tokens[1] == 0).all()
    assert probs[0, 0, 17] == 1.0 and probs[0, 0].sum() == 1.0


def test_greedy_ties_across_ctas_tensor_core():
    # The tensor-core kernel combines the CTAs' winners through 64-bit
    # decision keys (score bits above the complement of the index): equal
    # maxima held by different CTAs must resolve to the lowest index.  With
    # 313 tiles over the CTAs, tile t belongs to CTA t mod grid, so index
    # 20000 (tile 156) is reached before index 129 (tile 1) is finished.
    B, K, V, r = 6, 3, 40000, 64
    w = wl.make_custom(B, K, V, r, seed=21, base_dtype=wl.F32,
                       w_dtype=wl.BF16, w_std=0.0, greedy_rows=list(range(B)))
    w.base[:] = -1.0
    w.base[0, :, [39000, 20000, 129]] = 3.0   # three CTAs -> 129
    w.base[1, :, :] = 0.5                      # every CTA ties -> 0
    w.base[2, :, [6, 5]] = 2.0                 # one warp -> 5
    w.base[3, :, [39999, 39998, 38000]] = 7.0  # last tiles -> 38000
    w.base[4, 0, 777] = 4.0                    # a single maximum
    w.base[4, 1:, [31000, 30999]] = 4.0        # -> 30999
    w.base[5, :, 1:] = -np.inf                 # only index 0 finite -> 0
    tokens, logits, probs = _np(run_draft(w))
    ref = oracle.draft_block(w.base, w.U, w.Wb, w.d0, w.seed, w.offset, w.T,
                             greedy=w.greedy)
    np.testing.assert_array_equal(tokens, ref.tokens)
    assert list(tokens[:, 0]) == [129, 0, 5, 38000, 777, 0]
    assert (probs.sum(axis=2) == 1.0).all()   # one-hot proposals


def test_nan_valid_row_gives_legal_token():
    w = wl.make_custom(2, 2, 900, 16, seed=4)
    w.base[0, 0, ::3] = np.nan
    w.base[1, :, :] = np.nan  # a valid (non-padding) row of NaN
    tokens, logits, probs = _np(run_draft(w))
    assert ((tokens >= 0) & (tokens < w.V)).all()
    assert (tokens[1] == 0).all()
    ref = oracle.draft_block(w.base, w.U, w.Wb, w.d0, w.seed, w.offset, w.T)
    assert tokens[0, 0] == ref.tokens[0, 0]


# --------------------------------------------------------- determinism
def test_repeat_and_graph_replay_bitwise_and_new_offset():
    w = wl.make_custom(6, 4, 5000, 64, seed=9, base_dtype=wl.BF16,
                       w_dtype=wl.BF16, w_std=0.2, greedy_rows=[2])
    dev = to_device(w)
    ws = pkg.DraftWorkspace(w.B, w.K, w.V, w.r)
    eager1 = _np(run_draft(w, dev, workspace=ws))
    eager2 = _np(run_draft(w, dev, workspace=ws))
    for a, b in zip(eager1, eager2):
        np.testing.assert_array_equal(a, b)
    # CUDA-graph capture of the whole C-ABI call, then replay
    s = torch.cuda.Stream()
    outs = [torch.empty_like(t) for t in (torch.empty((w.B, w.K), dtype=torch.int32, device="cuda"),
                                          torch.empty((w.B, w.K, w.V), device="cuda"),
                                          torch.empty((w.B, w.K, w.V), device="cuda"))]
    call = lambda: pkg.draft_block(dev["base"], dev["U"], dev["Wb"], dev["d0"],
                                   dev["seed"], dev["offset"], w.T,
                                   greedy=dev["greedy"], tokens=outs[0],
                                   logits=outs[1], draft_probs=outs[2],
                                   workspace=ws, stream=s)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for t in outs:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager1, outs):
        np.testing.assert_array_equal(a, b.cpu().numpy())
    # a new offset draws anew (sampled rows), greedy row unchanged
    dev["offset"].add_(1)
    g.replay()
    torch.cuda.synchronize()
    t_new = outs[0].cpu().numpy()
    sampled = [b for b in range(w.B) if b != 2]
    assert (t_new[sampled] != eager1[0][sampled]).any()
    np.testing.assert_array_equal(t_new[2], eager1[0][2])


# ---------------------------------------------------------- distribution
def _chi2(tokens, probs):
    counts = np.bincount(tokens, minlength=len(probs)).astype(np.float64)
    exp = probs * counts.sum()
    keep = exp > 5
    c = np.append(counts[keep], counts[~keep].sum())
    e = np.append(exp[keep], exp[~keep].sum())
    if e[-1] == 0:
        c, e = c[:-1], e[:-1]
    return stats.chisquare(c, e).pvalue


@pytest.mark.parametrize("bdt", [wl.F32, wl.BF16])
def test_draws_follow_softmax_and_condition_on_previous(bdt):
    """Position 0 frequencies match softmax(l0 / T) and the joint (d0, d1)
    matches softmax(l0)[a] softmax(l1 | a)[b] (chi-square p = 1e-4), over
    many requests with distinct seeds, with the vocabulary split in several
    chunks."""
    V, r, K, T = 384, 16, 2, 0.9
    B, calls = 1024, 120
    rng = np.random.Generator(np.random.PCG64(int(bdt) + 5))
    base_rows = (rng.standard_normal((K, V)) * 0.6).astype(np.float32)
    base_rows[:, :6] += 3.0  # a few heavy tokens
    U = (rng.standard_normal((V, r)) * 0.6).astype(np.float32)
    Wb = (rng.standard_normal((r, V)) * 0.6).astype(np.float32)
    if bdt == wl.BF16:
        base_np = wl.to_bf16_bits(np.broadcast_to(base_rows, (B, K, V)).copy())
        base_f = wl.bf16_bits_to_f32(base_np[0])
    else:
        base_np = np.broadcast_to(base_rows, (B, K, V)).copy()
        base_f = base_rows
    w = wl.Workload("chi2", B, K, V, r, T, base_np, U, Wb,
                    np.full(B, 5, np.int32), np.zeros(B, np.uint64),
                    np.zeros(B, np.uint64))
    dev = to_device(w)
    toks = []
    for c in range(calls):
        dev["seed"].copy_(torch.arange(B, dtype=torch.int64) + c * B + 17)
        toks.append(run_draft(w, dev)[0].cpu().numpy())
    toks = np.concatenate(toks)
    U64, W64 = U.astype(np.float64), Wb.astype(np.float64)
    l0 = (base_f[0].astype(np.float64) + U64[5] @ W64).astype(np.float32)
    p0 = special.softmax((l0 / np.float32(T)).astype(np.float64))
    assert _chi2(toks[:, 0], p0) > 1e-4
    heavy = np.argsort(-p0)[:3]
    for a in heavy:  # position 1 given the drawn position 0
        l1 = (base_f[1].astype(np.float64) + U64[a] @ W64).astype(np.float32)
        p1 = special.softmax((l1 / np.float32(T)).astype(np.float64))
        m = toks[:, 0] == a
        assert _chi2(toks[m, 1], p1) > 1e-4


@pytest.mark.parametrize("V", [128, 384])
@pytest.mark.parametrize("bdt", [wl.F32, wl.BF16])
def test_tensor_core_draws_follow_softmax_and_condition_on_previous(V, bdt,
                                                                     monkeypatch):
    """The same chi-square tests (p = 1e-4) on the tensor-core kernel itself
    (bf16 head, r = 64): one vocab chunk (V = 128, one CTA) and three
    (V = 384, three CTAs whose winners meet through the decision keys), with
    f32 and bf16 drafter logits; position 0 against softmax(l0 / T) and
    position 1 given each of the three likeliest position-0 tokens."""
    monkeypatch.setenv("DSPARK_POSITION_KERNEL", "tc")  # fail if not taken
    r, K, T = 64, 2, 0.9
    B, calls = 96, 1300
    rng = np.random.Generator(np.random.PCG64(int(bdt) + 11 + V))
    base_rows = (rng.standard_normal((K, V)) * 0.6).astype(np.float32)
    base_rows[:, :6] += 3.0
    U_bits = wl.to_bf16_bits((rng.standard_normal((V, r)) * 0.4).astype(np.float32))
    Wb_bits = wl.to_bf16_bits((rng.standard_normal((r, V)) * 0.4).astype(np.float32))
    if bdt == wl.BF16:
        base_np = wl.to_bf16_bits(np.broadcast_to(base_rows, (B, K, V)).copy())
        base_f = wl.bf16_bits_to_f32(base_np[0])
    else:
        base_np = np.broadcast_to(base_rows, (B, K, V)).copy()
        base_f = base_rows
    w = wl.Workload("chi2_tc", B, K, V, r, T, base_np, U_bits, Wb_bits,
                    np.full(B, 5, np.int32), np.zeros(B, np.uint64),
                    np.zeros(B, np.uint64))
    dev = to_device(w)
    toks = []
    for c in range(calls):
        dev["seed"].copy_(torch.arange(B, dtype=torch.int64) + c * B + 29)
        toks.append(run_draft(w, dev)[0].cpu().numpy())
    toks = np.concatenate(toks)
    U64 = wl.bf16_bits_to_f32(U_bits).astype(np.float64)
    W64 = wl.bf16_bits_to_f32(Wb_bits).astype(np.float64)
    l0 = (base_f[0].astype(np.float64) + U64[5] @ W64).astype(np.float32)
    p0 = special.softmax((l0 / np.float32(T)).astype(np.float64))
    assert _chi2(toks[:, 0], p0) > 1e-4
    for a in np.argsort(-p0)[:3]:
        l1 = (base_f[1].astype(np.float64) + U64[a] @ W64).astype(np.float32)
        p1 = special.softmax((l1 / np.float32(T)).astype(np.float64))
        m = toks[:, 0] == a
        assert m.sum() > 2000
        assert _chi2(toks[m, 1], p1) > 1e-4
