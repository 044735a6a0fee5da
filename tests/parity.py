"""Parity helpers: move a synthetic workload to the GPU, run the C-ABI path,
and compare its outputs with the CPU oracle row by row.

Tolerances (the spec bar, with one derived widening):
  tokens       identical, except where the oracle's two best decision scores
               lie within 1e-5 of each other (a near tie that float32 noise or
               a one-ulp logit difference may resolve either way);
  logits       |gpu - oracle| <= 1e-6 + 1e-5 |oracle|;
  draft_probs  |gpu - oracle| <= 1e-6 + rtol_q |oracle| with
               rtol_q = max(1e-5, 4 ulp(max |s|)), s = l / T.  The kernels
               accumulate the bias in float32 while the oracle rounds a double
               once, so l may differ by one ulp; exp(s - M) then moves by
               ulp(l) / T relative, which for T >= 0.7 and |l| < 32 stays
               below 1e-5 and for small T (e.g. 0.05) needs the 4-ulp term.
  draft_probs  vs the row's own GPU logits (check_probs_against_own_logits):
               |q - softmax(float32(l / T))| <= 1e-6 + 1e-5 |ref| on every
               row, ref in double, no widening.
Comparisons are free-running: the oracle draws its own chain of every
request from d0 and never sees a GPU output.  Where the GPU's token at (b, k)
differs from the oracle's (allowed only at a near tie), the positions after
k of request b have other inputs on the two sides and are not compared;
such requests are counted.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
from ancestral_draft_sampling_gb300.workloads import to_device  # noqa: F401

TOKEN_TIE = 1e-5
LOGIT_ATOL, LOGIT_RTOL = 1e-6, 1e-5
PROB_ATOL, PROB_RTOL = 1e-6, 1e-5


def ulp32(x: float) -> float:
    x = abs(float(x))
    if x == 0 or not np.isfinite(x):
        return 2.0**-149
    return 2.0 ** (np.floor(np.log2(x)) - 23)


def prob_rtol(logits_row: np.ndarray, T: float) -> float:
    s = np.abs(logits_row[np.isfinite(logits_row)]) / T
    smax = float(s.max()) if s.size else 0.0
    return max(PROB_RTOL, 4 * ulp32(smax))


def default_rows(B, K, max_rows=None, seed=0):
    rows = [(b, k) for b in range(B) for k in range(K)]
    if max_rows is None or len(rows) <= max_rows:
        return rows
    first = [(b, 0) for b in range(B)]
    rest = [rk for rk in rows if rk[1] > 0]
    rng = np.random.Generator(np.random.PCG64(seed))
    pick = rng.choice(len(rest), size=max(0, max_rows - len(first)), replace=False)
    return sorted(first + [rest[i] for i in pick])


def check_block_against_oracle(w, tokens, logits, probs, rows=None,
                               threads=None):
    """Asserts parity of the GPU outputs (numpy) on `rows` (default: all).
    Each request's free-running oracle chain is drawn and compared in a
    worker thread (ctypes and numpy release the GIL), so that only a few
    rows of oracle output are alive at a time.  Returns a dict of counters
    (rows compared, near-tie token differences, rows skipped after such a
    difference)."""
    B, K, V = w.B, w.K, w.V
    rows = rows or default_rows(B, K)
    assert tokens.shape == (B, K)
    assert ((tokens >= 0) & (tokens < V)).all(), "token out of range"
    want = {}
    for b, k in rows:
        want.setdefault(b, set()).add(k)
    Ts = oracle.request_temperatures(w.T, B)  # w.T: scalar or per request

    def one(b):
        is_pad = bool(w.pad_row[b]) if w.pad_row is not None else False
        greedy = bool(w.greedy[b]) if w.greedy is not None else False
        prev = int(w.d0[b])
        checked = skipped = 0
        diverged = None
        for k in range(max(want[b]) + 1):
            o = oracle.draft_position(None if is_pad else w.base[b, k], w.U,
                                      w.Wb, prev, int(w.seed[b]),
                                      int(w.offset[b]), k, float(Ts[b]),
                                      greedy=greedy, is_pad=is_pad)
            where = f"(b={b}, k={k})"
            if k in want[b]:
                np.testing.assert_allclose(logits[b, k], o.logits,
                                           rtol=LOGIT_RTOL, atol=LOGIT_ATOL,
                                           equal_nan=True,
                                           err_msg=f"logits {where}")
                if greedy:
                    onehot = np.zeros(V, np.float32)
                    onehot[tokens[b, k]] = 1.0
                    np.testing.assert_array_equal(
                        probs[b, k], onehot, err_msg=f"greedy proposal {where}")
                else:
                    np.testing.assert_allclose(
                        probs[b, k], o.probs, atol=PROB_ATOL,
                        rtol=prob_rtol(o.logits, float(Ts[b])), equal_nan=True,
                        err_msg=f"draft_probs {where}")
                checked += 1
            if tokens[b, k] != o.token:
                gap = o.best - o.second
                assert gap <= TOKEN_TIE, (
                    f"token {where}: gpu {tokens[b, k]} oracle {o.token}, "
                    f"oracle top-2 gap {gap}")
                # later positions of b are conditioned on different tokens
                diverged = k
                skipped = sum(1 for kk in want[b] if kk > k)
                break
            prev = o.token
        return checked, skipped, diverged is not None

    todo = sorted(want)
    threads = threads or max(1, min(len(todo), os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        results = list(ex.map(one, todo))
    return {"rows": sum(r[0] for r in results),
            "near_tie_token_diffs": sum(1 for r in results if r[2]),
            "rows_after_divergence": sum(r[1] for r in results)}


def check_probs_against_own_logits(w, tokens, logits, probs):
    """The stored proposal of every row equals the softmax of the row's own
    float32 biased logits: s = logits / T is formed as the float32 IEEE
    quotient (the value the draw used, bit for bit) and the softmax is taken
    in double; |q - ref| <= 1e-6 + 1e-5 |ref| with no widening.  Greedy rows
    hold the one-hot of their token.  Returns the rows checked."""
    B, K, V = w.B, w.K, w.V
    Ts = oracle.request_temperatures(w.T, B)

    def one(b):
        greedy = w.greedy is not None and bool(w.greedy[b])
        for k in range(K):
            where = f"(b={b}, k={k})"
            if greedy:
                onehot = np.zeros(V, np.float32)
                onehot[tokens[b, k]] = 1.0
                np.testing.assert_array_equal(probs[b, k], onehot,
                                              err_msg=f"greedy proposal {where}")
                continue
            s = (logits[b, k] / np.float32(Ts[b])).astype(np.float64)
            s -= s.max()
            ref = np.exp(s)
            ref /= ref.sum()
            np.testing.assert_allclose(probs[b, k], ref, atol=PROB_ATOL,
                                       rtol=PROB_RTOL,
                                       err_msg=f"q vs own logits {where}")
        return K

    threads = max(1, min(B, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return sum(ex.map(one, range(B)))


def run_draft(w, dev=None, device="cuda:0", stream=None, workspace=None):
    import ancestral_draft_sampling_gb300 as pkg
    dev = dev or to_device(w, device)
    out = pkg.draft_block(dev["base"], dev["U"], dev["Wb"], dev["d0"],
                          dev["seed"], dev["offset"], w.T,
                          greedy=dev["greedy"], pad_row=dev["pad_row"],
                          workspace=workspace, stream=stream)
    torch.cuda.synchronize()
    return out
