"""The measurement entry points: dspark_draft_block_profile (CUDA events
around every launch) and dspark_draft_block_timeline (graph replay with
event nodes) compute the block itself -- the same outputs as
dspark_draft_block, bit for bit -- and report the launches they made."""
import numpy as np
import pytest
import torch

import ancestral_draft_sampling_gb300 as pkg
from ancestral_draft_sampling_gb300 import workloads as wl
from tests.parity import run_draft, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _outs(w):
    return (torch.empty((w.B, w.K), dtype=torch.int32, device="cuda"),
            torch.empty((w.B, w.K, w.V), device="cuda"),
            torch.empty((w.B, w.K, w.V), device="cuda"))


def _args(w, dev):
    return (dev["base"], dev["U"], dev["Wb"], dev["d0"], dev["seed"],
            dev["offset"], w.T)


@pytest.mark.parametrize("B,groups", [(40, 1), (150, 2)])
def test_profile_outputs_and_launch_counts(B, groups):
    w = wl.make_custom(B, 3, 8192, 128, seed=500 + B, base_dtype=wl.F32,
                       w_dtype=wl.BF16, w_std=0.2, greedy_rows=[1])
    dev = to_device(w)
    ref = [t.cpu().numpy() for t in run_draft(w, dev)]
    tok, lg, pr = _outs(w)
    stages = pkg.draft_block_profile(*_args(w, dev), greedy=dev["greedy"],
                                     pad_row=dev["pad_row"], tokens=tok,
                                     logits=lg, draft_probs=pr)
    for a, b in zip((tok, lg, pr), ref):
        np.testing.assert_array_equal(a.cpu().numpy(), b)
    # tensor-core kernel: K positions and one pick per request group, one
    # proposal writer for the block
    assert stages["position"][1] == groups * w.K
    assert stages["pick"][1] == groups
    assert stages["proposal"][1] == 1
    assert all(ms > 0.0 for ms, _ in stages.values())


@pytest.mark.parametrize("B", [40, 150])
def test_timeline_outputs_and_segments(B):
    w = wl.make_custom(B, 3, 8192, 128, seed=600 + B, base_dtype=wl.BF16,
                       w_dtype=wl.BF16, w_std=0.2)
    dev = to_device(w)
    ref = [t.cpu().numpy() for t in run_draft(w, dev)]
    tok, lg, pr = _outs(w)
    s = torch.cuda.Stream()
    chain, prop = pkg.draft_block_timeline(*_args(w, dev), replays=3, stream=s,
                                           tokens=tok, logits=lg,
                                           draft_probs=pr)
    for a, b in zip((tok, lg, pr), ref):
        np.testing.assert_array_equal(a.cpu().numpy(), b)
    assert chain > 0.0 and prop > 0.0
