"""dspark_draft_block_per_request: a temperature per request and
slot-indexed proposals (brb-nv/TensorRT-LLM PR #27, "2. One fused kernel per
draft position": the proposal writer stores q_k into the slot-indexed
draft_probs).  Each request must match the oracle run with its own
temperature. With equal temperatures the call must be bitwise
dspark_draft_block. Slots must receive exactly their request's proposals
and leave every other slot alone."""
import numpy as np
import pytest
import torch

import ancestral_draft_sampling_gb300 as pkg
from ancestral_draft_sampling_gb300 import workloads as wl
from tests.parity import check_block_against_oracle, run_draft, to_device

pytestmark = pytest.mark.gpu

TEMPS = [1.0, 0.7, 0.05, 20.0, 2.5, 1.0, 0.3, 1.5]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _temps(B, values=TEMPS):
    return np.array([values[b % len(values)] for b in range(B)], dtype=np.float32)


def _per_request(w, dev, temps, slot=None, draft_probs=None, workspace=None):
    t = torch.from_numpy(temps).cuda()
    s = None if slot is None else torch.from_numpy(slot.astype(np.int32)).cuda()
    out = pkg.draft_block_per_request(
        dev["base"], dev["U"], dev["Wb"], dev["d0"], dev["seed"], dev["offset"],
        t, greedy=dev["greedy"], pad_row=dev["pad_row"], slot=s,
        draft_probs=draft_probs, workspace=workspace)
    torch.cuda.synchronize()
    return [x.cpu().numpy() for x in out]


CASES = [
    # tensor-core kernel: bf16 head, greedy and padding requests
    dict(B=24, K=3, V=20000, r=256, seed=61, base_dtype=wl.F32,
         w_dtype=wl.BF16, greedy_rows=[3], pad_rows=[23], n_spikes=4),
    # tensor-core kernel with bf16 drafter logits (two staging tiles)
    dict(B=10, K=4, V=40000, r=128, seed=62, base_dtype=wl.BF16,
         w_dtype=wl.BF16),
    # bf16 drafter logits at B = 88, r = 256 (one staging tile)
    dict(B=88, K=2, V=8192, r=256, seed=66, base_dtype=wl.BF16,
         w_dtype=wl.BF16, greedy_rows=[2], pad_rows=[87]),
    # FFMA kernel: f32 head, ragged vocabulary
    dict(B=6, K=2, V=3001, r=32, seed=63, base_dtype=wl.F32, w_dtype=wl.F32),
    # 150 requests: two request groups of 75
    dict(B=150, K=2, V=8192, r=128, seed=69, base_dtype=wl.F32,
         w_dtype=wl.BF16, greedy_rows=[100], pad_rows=[149]),
]


@pytest.mark.parametrize("case", CASES)
def test_per_request_temperatures_match_oracle(case):
    c = dict(case)
    B, K, V, r = c.pop("B"), c.pop("K"), c.pop("V"), c.pop("r")
    w = wl.make_custom(B, K, V, r, w_std=0.2, **c)
    dev = to_device(w)
    temps = _temps(B)
    tokens, logits, probs = _per_request(w, dev, temps)
    w.T = temps  # the oracle runs each request with its own temperature
    st = check_block_against_oracle(w, tokens, logits, probs)
    assert st["near_tie_token_diffs"] <= 1


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_equal_temperatures_are_the_scalar_call(T):
    w = wl.make_custom(16, 3, 20000, 256, seed=64, base_dtype=wl.F32,
                       w_dtype=wl.BF16, w_std=0.2, greedy_rows=[5])
    w.T = T
    dev = to_device(w)
    ref = [x.cpu().numpy() for x in run_draft(w, dev)]
    got = _per_request(w, dev, np.full(w.B, T, dtype=np.float32))
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("B", [10, 130])  # 130: two request groups
def test_slots_receive_their_request_and_nothing_else(B):
    w = wl.make_custom(B, 3, 9000, 64, seed=65, base_dtype=wl.F32,
                       w_dtype=wl.BF16, w_std=0.2)
    dev = to_device(w)
    temps = _temps(w.B)
    _, _, plain = _per_request(w, dev, temps)
    rng = np.random.default_rng(66)
    n_slots = B + 6
    slot = rng.permutation(n_slots)[:w.B]
    buf = torch.full((n_slots, w.K, w.V), -1.0, device="cuda")
    _, _, got = _per_request(w, dev, temps, slot=slot, draft_probs=buf)
    for b in range(w.B):
        np.testing.assert_array_equal(got[slot[b]], plain[b])
    untouched = sorted(set(range(n_slots)) - set(slot.tolist()))
    assert (got[untouched] == -1.0).all()


def test_invalid_temperature_counts_as_one_and_is_reported():
    w = wl.make_custom(8, 2, 9000, 64, seed=67, base_dtype=wl.F32,
                       w_dtype=wl.BF16, w_std=0.2)
    dev = to_device(w)
    temps = _temps(w.B)
    bad = temps.copy()
    bad[2], bad[4], bad[6] = -1.0, np.nan, np.inf
    fixed = temps.copy()
    fixed[2] = fixed[4] = fixed[6] = 1.0
    ws = pkg.DraftWorkspace(w.B, w.K, w.V, w.r)
    ws.buffer.fill_(0xFF)  # stale contents: each call clears the error word
    got = _per_request(w, dev, bad, workspace=ws)
    assert pkg.read_device_error(ws) == 3
    ref = _per_request(w, dev, fixed, workspace=ws)
    assert pkg.read_device_error(ws) == 0
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a, b)


def test_slot_out_of_range_writes_nothing_and_is_reported():
    w = wl.make_custom(4, 2, 5000, 64, seed=68, base_dtype=wl.F32,
                       w_dtype=wl.BF16, w_std=0.2)
    dev = to_device(w)
    temps = _temps(w.B)
    _, _, plain = _per_request(w, dev, temps)
    slot = np.array([2, 9, 0, 1], dtype=np.int32)  # 9 is outside 5 slots
    buf = torch.full((5, w.K, w.V), -1.0, device="cuda")
    ws = pkg.DraftWorkspace(w.B, w.K, w.V, w.r)
    ws.buffer.fill_(0xFF)  # stale contents: each call clears the error word
    _, _, got = _per_request(w, dev, temps, slot=slot, draft_probs=buf,
                             workspace=ws)
    assert pkg.read_device_error(ws) == 4
    for b in (0, 2, 3):
        np.testing.assert_array_equal(got[slot[b]], plain[b])
    assert (got[[3, 4]] == -1.0).all()
