"""Seeded synthetic inputs for the draft-block sampler.

This module only draws random inputs; it holds none of the method's
arithmetic, so both the CUDA path's tests/bench and the CPU oracle can take
their inputs from it.

Shapes and distributions follow the drafting workload of brb-nv/TensorRT-LLM
PR #27, Results, "Drafting alone" (B x 7 x 200064 drafter logits, a rank-256
Markov head), with these recipes (the pages measure on SPEED-Bench serving
traffic; these synthetic inputs stand in for it):

  small   B=1,  K=3, V=4096,   r=64,  f32 base ~N(0,3^2), U,Wb f32 ~N(0,0.05^2),
          d0=17, T=1.0, seed=0, offset=0
  b8      B=8,  K=7, V=200064, r=256, bf16 base ~N(0,3^2) + 32 spikes of +12
          per (request, position) row, U,Wb bf16 ~N(0,0.02^2), d0 ~ U[0,V),
          T=1.0, seed[b]=1234+b, offset[b]=0
  b44     as b8 with B=44, T=0.7, requests 40..43 greedy
  b88     B=88, f32 base ~N(0,4^2) + spikes, U,Wb bf16 ~N(0,0.02^2), T=1.0,
          requests 80..87 are CUDA-graph padding rows whose base is NaN
  b64v    as b8 with B=64, plus target probabilities for verification:
          row k < K is softmax(base_k + N(0,1)), the bonus row K is
          softmax(base_{K-1} + N(0,1)) with fresh noise (float32)

The generator is numpy's PCG64 seeded with 1000 + config number; bfloat16
values are produced by round-to-nearest-even from float32 (torch's CPU
conversion) and carried as uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

F32, BF16 = 0, 1


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    K: int
    V: int
    r: int
    T: float
    base: np.ndarray            # [B,K,V] float32 or uint16 (bf16 bits)
    U: np.ndarray               # [V,r]
    Wb: np.ndarray              # [r,V]
    d0: np.ndarray              # [B] int32
    seed: np.ndarray            # [B] uint64
    offset: np.ndarray          # [B] uint64
    greedy: Optional[np.ndarray] = None   # [B] uint8
    pad_row: Optional[np.ndarray] = None  # [B] uint8
    target: Optional[np.ndarray] = None   # [B,K+1,V] float32

    @property
    def base_dtype(self) -> int:
        return F32 if self.base.dtype == np.float32 else BF16

    @property
    def w_dtype(self) -> int:
        return F32 if self.U.dtype == np.float32 else BF16

    def base_f32(self) -> np.ndarray:
        return self.base if self.base.dtype == np.float32 else bf16_bits_to_f32(self.base)


def _normal(rng, shape, std, dtype=np.float32):
    out = rng.standard_normal(size=shape, dtype=np.float32)
    out *= np.float32(std)
    return out.astype(dtype, copy=False)


def _spike(rng, base: np.ndarray, n_spikes: int, height: float) -> None:
    """Add `height` at n_spikes distinct uniform indices of every row."""
    B, K, V = base.shape
    flat = base.reshape(B * K, V)
    for row in range(B * K):
        idx = rng.choice(V, size=n_spikes, replace=False)
        flat[row, idx] += np.float32(height)


def make_custom(B, K, V, r, *, seed=1, base_std=3.0, w_std=0.02,
                base_dtype=F32, w_dtype=F32, T=1.0, n_spikes=0,
                spike=12.0, greedy_rows=(), pad_rows=(), nan_pad=True,
                req_seed0=1234, offset=0, d0=None, target=False) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed))
    base = _normal(rng, (B, K, V), base_std)
    if n_spikes:
        _spike(rng, base, n_spikes, spike)
    U = _normal(rng, (V, r), w_std)
    Wb = _normal(rng, (r, V), w_std)
    if d0 is None:
        d0 = rng.integers(0, V, size=B, dtype=np.int64).astype(np.int32)
    else:
        d0 = np.broadcast_to(np.asarray(d0, dtype=np.int32), (B,)).copy()
    greedy = None
    if len(greedy_rows):
        greedy = np.zeros(B, dtype=np.uint8)
        greedy[list(greedy_rows)] = 1
    pad = None
    if len(pad_rows):
        pad = np.zeros(B, dtype=np.uint8)
        pad[list(pad_rows)] = 1
        if nan_pad:
            base[list(pad_rows)] = np.nan
    tgt = None
    if target:
        noise = _normal(rng, (B, K + 1, V), 1.0)
        logits = np.concatenate([base, base[:, K - 1:K]], axis=1) + noise
        logits = logits.astype(np.float64)
        logits -= logits.max(axis=2, keepdims=True)
        np.exp(logits, out=logits)
        logits /= logits.sum(axis=2, keepdims=True)
        tgt = logits.astype(np.float32)
    if base_dtype == BF16:
        base = to_bf16_bits(base)
    if w_dtype == BF16:
        U = to_bf16_bits(U)
        Wb = to_bf16_bits(Wb)
    seeds = (np.arange(B, dtype=np.uint64) + np.uint64(req_seed0))
    offs = np.full(B, offset, dtype=np.uint64)
    return Workload(name=f"custom_B{B}_K{K}_V{V}_r{r}", B=B, K=K, V=V, r=r,
                    T=float(T), base=base, U=U, Wb=Wb, d0=d0, seed=seeds,
                    offset=offs, greedy=greedy, pad_row=pad, target=tgt)


@dataclasses.dataclass
class VerifyInputs:
    """Inputs of standard verification for B requests of K drafts."""
    B: int
    K: int
    V: int
    q: np.ndarray        # [B,K,V] float32: the proposals the drafts came from
    p: np.ndarray        # [B,K+1,V] float32: the target's distributions
    tokens: np.ndarray   # [B,K] int32: drafts, token k drawn from q[b,k]
    seed: np.ndarray     # [B] uint64
    offset: np.ndarray   # [B] uint64


def _softmax_rows(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float64)
    x -= x.max(axis=-1, keepdims=True)
    np.exp(x, out=x)
    x /= x.sum(axis=-1, keepdims=True)
    return x


def make_verify(B, K, V, *, seed=1, logit_std=3.0, target_noise=1.0,
                n_spikes=32, spike=12.0, req_seed0=1234,
                offset=0) -> VerifyInputs:
    """Synthetic verification inputs: per request, drafter logits
    ~N(0, logit_std^2) plus n_spikes spikes per row; q = softmax of them;
    target row k < K = softmax(logits_k + N(0, target_noise^2)), the bonus
    row K = softmax(logits_{K-1} + fresh noise); draft k is drawn from q_k
    by numpy's generator (inverse CDF), so acceptance rates are those of a
    drafter that is this close to the target."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = np.empty((B, K, V), dtype=np.float32)
    p = np.empty((B, K + 1, V), dtype=np.float32)
    tokens = np.empty((B, K), dtype=np.int32)
    for b in range(B):  # one request at a time keeps the float64 rows small
        logits = _normal(rng, (1, K, V), logit_std)
        if n_spikes:
            _spike(rng, logits, min(n_spikes, V), spike)
        logits = logits[0]
        qb = _softmax_rows(logits)
        q[b] = qb
        tgt = np.concatenate([logits, logits[K - 1:K]], axis=0)
        tgt = tgt + _normal(rng, (K + 1, V), target_noise)
        p[b] = _softmax_rows(tgt)
        cdf = np.cumsum(qb, axis=1)
        u = rng.random(K) * cdf[:, -1]
        for k in range(K):
            tokens[b, k] = min(int(np.searchsorted(cdf[k], u[k], side="right")),
                               V - 1)
    seeds = np.arange(B, dtype=np.uint64) + np.uint64(req_seed0)
    offs = np.full(B, offset, dtype=np.uint64)
    return VerifyInputs(B=B, K=K, V=V, q=q, p=p, tokens=tokens, seed=seeds,
                        offset=offs)


def _tensor(a: np.ndarray, device):
    """numpy -> torch on `device`: bf16 bit patterns (uint16) become
    bfloat16 and uint64 becomes int64 with the same bits."""
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    if a.dtype == np.uint64:
        return torch.from_numpy(a.view(np.int64)).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_device(w: Workload, device="cuda:0") -> dict:
    """The workload's arrays as torch tensors on `device`, in the dtypes the
    binding takes (base, U, Wb, d0 int32, seed/offset int64, greedy/pad_row
    uint8 or None, and target when the workload has one)."""
    d = {
        "base": _tensor(w.base, device),
        "U": _tensor(w.U, device),
        "Wb": _tensor(w.Wb, device),
        "d0": _tensor(w.d0.astype(np.int32), device),
        "seed": _tensor(w.seed, device),
        "offset": _tensor(w.offset, device),
        "greedy": None if w.greedy is None else _tensor(w.greedy, device),
        "pad_row": None if w.pad_row is None else _tensor(w.pad_row, device),
    }
    if w.target is not None:
        d["target"] = _tensor(w.target, device)
    return d


CONFIG_NAMES = {1: "small", 2: "b8", 3: "b44", 4: "b88", 5: "b64v"}


def make_config(i: int) -> Workload:
    """The five configurations described in the module docstring."""
    vocab, rank = 200064, 256
    if i == 1:
        w = make_custom(1, 3, 4096, 64, seed=1001, base_std=3.0, w_std=0.05,
                        base_dtype=F32, w_dtype=F32, T=1.0, d0=17,
                        req_seed0=0, offset=0)
    elif i == 2:
        w = make_custom(8, 7, vocab, rank, seed=1002, base_std=3.0,
                        w_std=0.02, base_dtype=BF16, w_dtype=BF16, T=1.0,
                        n_spikes=32)
    elif i == 3:
        w = make_custom(44, 7, vocab, rank, seed=1003, base_std=3.0,
                        w_std=0.02, base_dtype=BF16, w_dtype=BF16, T=0.7,
                        n_spikes=32, greedy_rows=range(40, 44))
    elif i == 4:
        w = make_custom(88, 7, vocab, rank, seed=1004, base_std=4.0,
                        w_std=0.02, base_dtype=F32, w_dtype=BF16, T=1.0,
                        n_spikes=32, pad_rows=range(80, 88))
    elif i == 5:
        w = make_custom(64, 7, vocab, rank, seed=1005, base_std=3.0,
                        w_std=0.02, base_dtype=BF16, w_dtype=BF16, T=1.0,
                        n_spikes=32, target=True)
    else:
        raise ValueError(f"no configuration {i}")
    w.name = CONFIG_NAMES[i]
    return w
