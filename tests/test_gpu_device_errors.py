"""The device error word of the draft-block workspace, on the GPU.

Every call clears the word when it starts (one memset with the decision
keys), so a workspace full of stale bytes reads 0 after a clean call; a d0
outside [0, V) is replaced by token 0 and reported as code 1; and a bounded
wait that runs out is reported as code 2 while the context stays usable.
The failure is made on purpose only in the last form the failure-detection
rules allow: a wait on a barrier phase that nothing completes (it guards no
copy), with a short limit, on a small shape."""
import numpy as np
import pytest
import torch

import ancestral_draft_sampling_gb300 as pkg
from ancestral_draft_sampling_gb300 import workloads as wl
from tests.parity import check_block_against_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _np(out):
    return tuple(t.cpu().numpy() for t in out)


def _call(w, dev, ws):
    out = pkg.draft_block(dev["base"], dev["U"], dev["Wb"], dev["d0"],
                          dev["seed"], dev["offset"], w.T, greedy=dev["greedy"],
                          pad_row=dev["pad_row"], workspace=ws)
    torch.cuda.synchronize()
    return _np(out)


# the tensor-core kernel (bf16 head, r % 16 == 0, V % 8 == 0) and the FFMA one
CASES = {
    "tensor_core": dict(B=6, K=3, V=4096, r=64, w_dtype=wl.BF16, kernel="tc"),
    "ffma": dict(B=5, K=3, V=3001, r=32, w_dtype=wl.F32, kernel="generic"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_clean_call_on_stale_workspace_reads_no_error(name, monkeypatch):
    c = CASES[name]
    monkeypatch.setenv("DSPARK_POSITION_KERNEL", c["kernel"])
    w = wl.make_custom(c["B"], c["K"], c["V"], c["r"], seed=81,
                       w_dtype=c["w_dtype"], w_std=0.2, greedy_rows=[1])
    dev = to_device(w)
    ws = pkg.DraftWorkspace(w.B, w.K, w.V, w.r)
    for _ in range(2):  # a fresh-looking workspace, twice in a row
        ws.buffer.fill_(0xFF)
        tokens, logits, probs = _call(w, dev, ws)
        assert pkg.read_device_error(ws) == 0
    st = check_block_against_oracle(w, tokens, logits, probs)
    assert st["near_tie_token_diffs"] <= 1


@pytest.mark.parametrize("name", sorted(CASES))
def test_bad_d0_draws_from_token_zero_and_is_reported(name, monkeypatch):
    """A d0 outside [0, V) is replaced by 0 (device error 1): the request's
    chain is then the oracle's chain from d0 = 0, and the other requests are
    unaffected."""
    c = CASES[name]
    monkeypatch.setenv("DSPARK_POSITION_KERNEL", c["kernel"])
    w = wl.make_custom(c["B"], c["K"], c["V"], c["r"], seed=82,
                       w_dtype=c["w_dtype"], w_std=0.3)
    w.d0[1] = -5
    w.d0[3] = w.V + 3
    dev = to_device(w)
    ws = pkg.DraftWorkspace(w.B, w.K, w.V, w.r)
    tokens, logits, probs = _call(w, dev, ws)
    assert pkg.read_device_error(ws) == 1
    w.d0[1] = 0
    w.d0[3] = 0
    st = check_block_against_oracle(w, tokens, logits, probs)
    assert st["near_tie_token_diffs"] <= 1
    # the next call with legal inputs is clean and gives the same outputs
    dev["d0"].copy_(torch.from_numpy(w.d0))
    again = _call(w, dev, ws)
    assert pkg.read_device_error(ws) == 0
    for a, b in zip(again, (tokens, logits, probs)):
        np.testing.assert_array_equal(a, b)


def test_wait_that_runs_out_reports_timeout_and_context_stays_usable(monkeypatch):
    """DSPARK_TEST_STALL_WAIT=1 makes the tensor-core kernel's MMA issuer
    wait on a barrier phase that nothing completes, with a short poll limit.
    The kernel records code 2, stops issuing, lets its issued copies land,
    frees its tensor memory and returns; the next call, without the stall,
    is clean and matches the oracle."""
    monkeypatch.setenv("DSPARK_POSITION_KERNEL", "tc")
    w = wl.make_custom(4, 1, 1024, 64, seed=83, w_dtype=wl.BF16, w_std=0.2)
    dev = to_device(w)
    ws = pkg.DraftWorkspace(w.B, w.K, w.V, w.r)
    monkeypatch.setenv("DSPARK_TEST_STALL_WAIT", "1")
    _call(w, dev, ws)
    assert pkg.read_device_error(ws) == 2
    monkeypatch.delenv("DSPARK_TEST_STALL_WAIT")
    tokens, logits, probs = _call(w, dev, ws)
    assert pkg.read_device_error(ws) == 0
    st = check_block_against_oracle(w, tokens, logits, probs)
    assert st["near_tie_token_diffs"] == 0


def test_host_fed_call_clears_the_error_word():
    w = wl.make_custom(4, 2, 4096, 64, seed=84, w_dtype=wl.BF16, w_std=0.2)
    dev = to_device(w)
    ws = pkg.HostWorkspace(w.B, w.K, w.V, w.r)
    ws.buffer.fill_(0xFF)
    host = lambda a: wl._tensor(a, "cpu").pin_memory()
    logits = torch.empty((w.B, w.K, w.V), device="cuda")
    probs = torch.empty_like(logits)
    base_dev = torch.empty_like(dev["base"])
    copy_stream = torch.cuda.Stream()
    pkg.draft_block_host(host(w.base), dev["U"], dev["Wb"],
                         host(w.d0.astype(np.int32)), host(w.seed),
                         host(w.offset), w.T, base_dev=base_dev, logits=logits,
                         draft_probs=probs, workspace=ws,
                         copy_stream=copy_stream)
    torch.cuda.synchronize()
    assert pkg.read_device_error(ws) == 0
