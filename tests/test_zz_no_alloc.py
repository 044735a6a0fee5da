"""dspark_draft_block_noalloc: the draft block for callers that cannot
allocate device memory (they are handed only their input and output buffers
by a host runtime that owns all device memory, or run where cudaMalloc must
not be called).  Its scratch is a library-owned device array instead of a
caller workspace; its outputs must equal the workspace entry point's.

The file is named to be collected last: a run that stops at the first
failure has already run every other test.  It passes alone in a fresh
process as well as after the other tests."""
import numpy as np
import pytest
import torch

import ancestral_draft_sampling_gb300 as pkg
from ancestral_draft_sampling_gb300 import workloads as wl
from ancestral_draft_sampling_gb300.workloads import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _outputs(w, device="cuda"):
    return (torch.empty((w.B, w.K), dtype=torch.int32, device=device),
            torch.empty((w.B, w.K, w.V), dtype=torch.float32, device=device),
            torch.empty((w.B, w.K, w.V), dtype=torch.float32, device=device))


def _compare(got, want):
    # the same launch sequence on the same inputs: bit-identical outputs
    for g, r in zip(got, want):
        np.testing.assert_array_equal(g.cpu().numpy(), r.cpu().numpy())


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    cases = [
        # tensor-core path: bf16 head, r % 16 == 0, V % 8 == 0
        wl.make_custom(40, 3, 20000, 256, seed=71, base_dtype=wl.F32,
                       w_dtype=wl.BF16, w_std=0.2, greedy_rows=[3],
                       pad_rows=[39], n_spikes=4),
        # FFMA path: float32 head, ragged vocabulary
        wl.make_custom(5, 2, 3001, 32, seed=72, base_dtype=wl.BF16,
                       w_dtype=wl.F32, w_std=0.2, T=0.8),
    ]
    for w in cases:
        dev = to_device(w)
        ref = pkg.draft_block(dev["base"], dev["U"], dev["Wb"], dev["d0"],
                              dev["seed"], dev["offset"], w.T,
                              greedy=dev["greedy"], pad_row=dev["pad_row"])
        for _ in range(2):  # two calls in a row share the scratch
            out = pkg.draft_block_noalloc(
                dev["base"], dev["U"], dev["Wb"], dev["d0"], dev["seed"],
                dev["offset"], w.T, greedy=dev["greedy"],
                pad_row=dev["pad_row"], tokens=_outputs(w)[0])
            torch.cuda.synchronize()
            _compare(out, ref)
        # a new offset through the scratch still matches the workspace path
        dev["offset"].add_(1)
        ref2 = pkg.draft_block(dev["base"], dev["U"], dev["Wb"], dev["d0"],
                               dev["seed"], dev["offset"], w.T,
                               greedy=dev["greedy"], pad_row=dev["pad_row"])
        out2 = pkg.draft_block_noalloc(dev["base"], dev["U"], dev["Wb"],
                                       dev["d0"], dev["seed"], dev["offset"],
                                       w.T, greedy=dev["greedy"],
                                       pad_row=dev["pad_row"])
        torch.cuda.synchronize()
        _compare(out2, ref2)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # B = 200, K = 7 needs ~3.2 MiB of scratch: refused before any launch
    B, K, V, r = 200, 7, 1024, 64
    assert pkg.workspace_bytes(B, K, V, r) > 2 << 20
    base = torch.zeros((B, K, V), dtype=torch.float32, device="cuda")
    U = torch.zeros((V, r), dtype=torch.float32, device="cuda")
    Wb = torch.zeros((r, V), dtype=torch.float32, device="cuda")
    d0 = torch.zeros(B, dtype=torch.int32, device="cuda")
    seed = torch.zeros(B, dtype=torch.int64, device="cuda")
    with pytest.raises(pkg.DsparkError) as err:
        pkg.draft_block_noalloc(base, U, Wb, d0, seed, seed, 1.0)
    assert err.value.status == 3  # DSPARK_ERR_WORKSPACE
