"""dspark_draft_block_host: the draft block with its inputs in pinned host
memory and the tokens returned to host memory.  The call copies each
position's drafter logits on a second stream while earlier positions
compute, and writes each position's proposals right after its pick; its
outputs must be bitwise those of dspark_draft_block on the same inputs
(the same kernels run on the same values), eagerly and from a CUDA graph."""
import numpy as np
import pytest
import torch

import ancestral_draft_sampling_gb300 as pkg
from ancestral_draft_sampling_gb300 import workloads as wl
from ancestral_draft_sampling_gb300.workloads import _tensor as _t
from tests.parity import run_draft, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _host(a):
    return _t(a, "cpu").pin_memory()


def _host_inputs(w):
    return dict(base=_host(w.base), d0=_host(w.d0.astype(np.int32)),
                seed=_host(w.seed), offset=_host(w.offset),
                greedy=None if w.greedy is None else _host(w.greedy),
                pad=None if w.pad_row is None else _host(w.pad_row))


def _host_call(w, dev, h, stream, copy_stream, ws=None, base_dev=None,
               out=None):
    B, K, V = w.B, w.K, w.V
    if base_dev is None:
        base_dev = torch.empty_like(dev["base"])
    if out is None:
        out = (torch.empty((B, K, V), dtype=torch.float32, device="cuda"),
               torch.empty((B, K, V), dtype=torch.float32, device="cuda"),
               torch.empty((B, K), dtype=torch.int32).pin_memory())
    logits, probs, tok_h = out
    pkg.draft_block_host(h["base"], dev["U"], dev["Wb"], h["d0"], h["seed"],
                         h["offset"], w.T, base_dev=base_dev, logits=logits,
                         draft_probs=probs, tokens_host=tok_h,
                         greedy_host=h["greedy"], pad_row_host=h["pad"],
                         workspace=ws, stream=stream, copy_stream=copy_stream)
    return tok_h, logits, probs


CASES = [
    # tensor-core path: bf16 head, f32 logits, greedy and padding requests
    dict(B=40, K=3, V=20000, r=256, seed=81, base_dtype=wl.F32,
         w_dtype=wl.BF16, greedy_rows=[5], pad_rows=[39], n_spikes=4),
    # tensor-core path with bf16 logits and T != 1
    dict(B=16, K=4, V=40000, r=128, seed=82, base_dtype=wl.BF16,
         w_dtype=wl.BF16, T=0.7),
    # bf16 logits at B = 72, r = 256 (one staging tile)
    dict(B=72, K=2, V=6144, r=256, seed=85, base_dtype=wl.BF16,
         w_dtype=wl.BF16),
    # FFMA path: f32 head, ragged vocabulary
    dict(B=5, K=2, V=3001, r=32, seed=83, base_dtype=wl.F32, w_dtype=wl.F32),
    # 130 requests: two request groups, each position's proposals per group
    dict(B=130, K=3, V=4096, r=64, seed=86, base_dtype=wl.F32,
         w_dtype=wl.BF16, greedy_rows=[70]),
]


@pytest.mark.parametrize("case", CASES)
def test_host_feed_equals_device_call(case):
    c = dict(case)
    B, K, V, r = c.pop("B"), c.pop("K"), c.pop("V"), c.pop("r")
    w = wl.make_custom(B, K, V, r, w_std=0.2, **c)
    dev = to_device(w)
    ref_tok, ref_logits, ref_probs = run_draft(w, dev)
    stream = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    h = _host_inputs(w)
    tok_h, logits, probs = _host_call(w, dev, h, stream, copy_stream)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tok_h.numpy(), ref_tok.cpu().numpy())
    assert torch.equal(logits, ref_logits)
    assert torch.equal(probs, ref_probs)


def test_host_feed_graph_replay():
    w = wl.make_custom(24, 3, 20000, 256, seed=84, base_dtype=wl.F32,
                       w_dtype=wl.BF16, w_std=0.2, n_spikes=4)
    dev = to_device(w)
    ref_tok, ref_logits, ref_probs = run_draft(w, dev)
    side, copy_stream = torch.cuda.Stream(), torch.cuda.Stream()
    ws = pkg.HostWorkspace(w.B, w.K, w.V, w.r)
    base_dev = torch.empty_like(dev["base"])
    out = (torch.empty_like(ref_logits), torch.empty_like(ref_probs),
           torch.empty((w.B, w.K), dtype=torch.int32).pin_memory())
    h = _host_inputs(w)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside capture
        _host_call(w, dev, h, side, copy_stream, ws, base_dev, out)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
        _host_call(w, dev, h, side, copy_stream, ws, base_dev, out)
    for _ in range(2):
        out[2].zero_()
        out[0].zero_()
        graph.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out[2].numpy(), ref_tok.cpu().numpy())
        assert torch.equal(out[0], ref_logits)
        assert torch.equal(out[1], ref_probs)
