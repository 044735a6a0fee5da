"""Parity of dspark_sample_temperature (temperature-only target sampling,
brb-nv/TensorRT-LLM PR #27, "1. Temperature-only sampling runs no filter")
with the CPU oracle.  Tokens must be identical except where the oracle's two
best scores lie within TOKEN_TIE of each other. Probabilities must meet the
proposal tolerance of the draft block (the same softmax arithmetic)."""
import types

import numpy as np
import pytest
import torch

import ancestral_draft_sampling_gb300 as pkg
import oracle
from tests.parity import PROB_ATOL, TOKEN_TIE, prob_rtol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _rows(R, V, seed, std=3.0, spikes=8):
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, std, (R, V)).astype(np.float32)
    for i in range(R):
        x[i, rng.choice(V, size=min(spikes, V), replace=False)] += 10.0
    s = rng.integers(0, 2**63, R, dtype=np.uint64)
    o = rng.integers(0, 2**40, R, dtype=np.uint64)
    return x, s, o


def _u64(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int64)).cuda()


def _gpu(x, s, o, T=1.0, temperature=None, greedy=None, position=None,
         with_probs=True, workspace=None):
    dev = lambda a, dt: None if a is None else torch.from_numpy(
        np.ascontiguousarray(a).astype(dt)).cuda()
    tok, probs = pkg.sample_temperature(
        torch.from_numpy(x).cuda(), _u64(s), _u64(o), T=T,
        temperature=dev(temperature, np.float32), greedy=dev(greedy, np.uint8),
        position=dev(position, np.int32), with_probs=with_probs,
        workspace=workspace)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), None if probs is None else probs.cpu().numpy()


def _check(x, s, o, tok, probs, T, greedy=None, position=None):
    ref = oracle.sample_temperature(x, T, s, o, greedy=greedy, position=position)
    Ts = oracle.request_temperatures(T, len(x))
    diffs = 0
    for i in range(len(x)):
        if tok[i] != ref.tokens[i]:
            gap = float(ref.top2[i, 0] - ref.top2[i, 1])
            assert gap <= TOKEN_TIE, f"row {i}: gpu {tok[i]} oracle {ref.tokens[i]}"
            diffs += 1
            continue
        if probs is not None:
            np.testing.assert_allclose(probs[i], ref.probs[i], atol=PROB_ATOL,
                                       rtol=prob_rtol(x[i], float(Ts[i])),
                                       err_msg=f"probs row {i}")
    return diffs


@pytest.mark.parametrize("R,V,T", [
    (16, 5001, 1.0),      # ragged vocabulary (scalar loads), many chunks
    (64, 40000, 0.7),     # float4 loads, T != 1
    (3, 200064, 1.0),     # the full vocabulary, few rows
    (700, 1024, 1.3),     # many rows, one chunk each
])
def test_sampler_matches_oracle(R, V, T):
    x, s, o = _rows(R, V, seed=R + V)
    tok, probs = _gpu(x, s, o, T=T)
    assert _check(x, s, o, tok, probs, T) <= 1


def test_sampler_per_row_temperatures_greedy_and_positions():
    R, V = 40, 20000
    x, s, o = _rows(R, V, seed=5)
    temps = np.array([[0.5, 1.0, 2.0, 0.05][i % 4] for i in range(R)], np.float32)
    greedy = np.zeros(R, np.uint8)
    greedy[[3, 17]] = 1
    x[17, [11, 12000]] = 40.0                       # a greedy tie: index 11
    pos = np.arange(R, dtype=np.int32) % 9
    tok, probs = _gpu(x, s, o, temperature=temps, greedy=greedy, position=pos)
    assert _check(x, s, o, tok, probs, temps, greedy=greedy, position=pos) <= 1
    assert tok[17] == 11 and probs[17, 11] == 1.0 and probs[17].sum() == 1.0


def test_sampler_tokens_only_and_deterministic():
    x, s, o = _rows(32, 30000, seed=6)
    t1, p1 = _gpu(x, s, o, T=0.9)
    t2, p2 = _gpu(x, s, o, T=0.9)
    t3, p3 = _gpu(x, s, o, T=0.9, with_probs=False)
    np.testing.assert_array_equal(t1, t2)
    np.testing.assert_array_equal(p1, p2)
    np.testing.assert_array_equal(t1, t3)
    assert p3 is None


def test_sampler_reports_bad_temperature_and_position():
    R, V = 6, 4096
    x, s, o = _rows(R, V, seed=7)
    nbytes = pkg._lib.load().dspark_sample_workspace_bytes(R, V)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    handle = types.SimpleNamespace(buffer=ws)
    ws.fill_(0xFF)  # stale contents: each call clears the error word
    temps = np.ones(R, np.float32)
    temps[2] = -3.0
    tok, _ = _gpu(x, s, o, temperature=temps, workspace=ws)
    assert pkg.read_device_error(handle) == 3
    ws.fill_(0xFF)
    ref, _ = _gpu(x, s, o, temperature=np.ones(R, np.float32), workspace=ws)
    assert pkg.read_device_error(handle) == 0
    np.testing.assert_array_equal(tok, ref)
    pos = np.zeros(R, np.int32)
    pos[4] = 70000
    _gpu(x, s, o, position=pos, workspace=ws)
    assert pkg.read_device_error(handle) == 5
