"""GB300-native DSpark ancestral draft-block sampling.

The sampler of brb-nv/TensorRT-LLM PR #27 ("2. One fused kernel per draft
position") with the semantics of brb-nv/TensorRT-LLM PR #21 ("2. Golden
sampling semantics"), as hand-written CUDA for sm_103a behind the C ABI in
``include/dspark.h``.  This module is the thin PyTorch-facing binding: it
takes torch tensors, checks dtypes and shapes, and passes raw pointers and
the current CUDA stream to the library.
"""
from __future__ import annotations

import ctypes
from typing import Optional

from . import _lib
from ._lib import BF16, F32, DsparkError  # noqa: F401

__all__ = ["draft_block", "draft_block_per_request", "draft_block_noalloc",
           "draft_block_profile", "draft_block_timeline", "sample_temperature",
           "draft_block_host", "HostWorkspace", "verify_standard", "verify_block",
           "noise_words", "workspace_bytes", "read_device_error",
           "DraftWorkspace", "DsparkError", "F32", "BF16", "version"]


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"expected float32 or bfloat16, got {t.dtype}")


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def version() -> str:
    return _lib.load().dspark_version().decode()


def workspace_bytes(B: int, K: int, V: int, r: int) -> int:
    return int(_lib.load().dspark_draft_workspace_bytes(B, K, V, r))


class DraftWorkspace:
    """Device scratch for dspark_draft_block, sized for (B, K, V, r)."""

    def __init__(self, B: int, K: int, V: int, r: int, device=None):
        torch = _torch()
        n = workspace_bytes(B, K, V, r)
        if n == 0:
            raise DsparkError("dspark_draft_workspace_bytes", 2)
        self.nbytes = n
        # torch's caching allocator returns 512-byte aligned blocks
        self.buffer = torch.empty(n, dtype=torch.uint8,
                                  device=device or "cuda")


def _check_draft_inputs(base_logits, U, Wb, d0, seed, offset, greedy,
                        pad_row, tokens=None, logits=None, draft_probs=None):
    """Shapes, dtypes and contiguity of draft_block's tensors; returns
    (B, K, V, r)."""
    torch = _torch()
    if base_logits.dim() != 3:
        raise ValueError("base_logits must be [B, K, V]")
    B, K, V = base_logits.shape
    if U.dim() != 2:
        raise ValueError("U must be [V, r]")
    r = U.shape[1]
    if tuple(U.shape) != (V, r) or tuple(Wb.shape) != (r, V):
        raise ValueError("U must be [V, r] and Wb [r, V]")
    if U.dtype != Wb.dtype:
        raise TypeError("U and Wb must share a dtype")
    _dtype_code(base_logits)
    _dtype_code(U)
    if d0.dtype != torch.int32 or tuple(d0.shape) != (B,):
        raise TypeError("d0 must be int32 [B]")
    for name, t in (("seed", seed), ("offset", offset)):
        if t.dtype != torch.int64 or tuple(t.shape) != (B,):
            raise TypeError(f"{name} must be int64 [B] (uint64 bit patterns)")
    for name, t in (("greedy", greedy), ("pad_row", pad_row)):
        if t is not None and (t.dtype != torch.uint8 or tuple(t.shape) != (B,)):
            raise TypeError(f"{name} must be uint8 [B] or None")
    if tokens is not None and (tokens.dtype != torch.int32 or
                               tuple(tokens.shape) != (B, K)):
        raise TypeError("tokens must be int32 [B, K]")
    for name, t in (("logits", logits), ("draft_probs", draft_probs)):
        if t is not None and (t.dtype != torch.float32 or
                              tuple(t.shape) != (B, K, V)):
            raise TypeError(f"{name} must be float32 [B, K, V]")
    for t in (base_logits, U, Wb, d0, seed, offset, greedy, pad_row, tokens,
              logits, draft_probs):
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    return B, K, V, r


def draft_block(base_logits, U, Wb, d0, seed, offset, T: float, *,
                greedy=None, pad_row=None, tokens=None, logits=None,
                draft_probs=None, workspace: Optional[DraftWorkspace] = None,
                stream=None):
    """Drafts one K-token block for B requests.  See include/dspark.h.

    base_logits [B,K,V] float32|bfloat16, U [V,r], Wb [r,V] (same dtype),
    d0 [B] int32, seed/offset [B] int64 (bit patterns of uint64),
    greedy/pad_row [B] uint8 or None.  Returns (tokens, logits, draft_probs).
    """
    torch = _torch()
    B, K, V, r = _check_draft_inputs(base_logits, U, Wb, d0, seed, offset,
                                     greedy, pad_row, tokens, logits,
                                     draft_probs)
    dev = base_logits.device
    if tokens is None:
        tokens = torch.empty((B, K), dtype=torch.int32, device=dev)
    if logits is None:
        logits = torch.empty((B, K, V), dtype=torch.float32, device=dev)
    if draft_probs is None:
        draft_probs = torch.empty((B, K, V), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = DraftWorkspace(B, K, V, r, device=dev)
    st = _lib.load().dspark_draft_block(
        _ptr(base_logits), _dtype_code(base_logits), _ptr(U), _ptr(Wb),
        _dtype_code(U), _ptr(d0), _ptr(seed), _ptr(offset), float(T),
        _ptr(greedy), _ptr(pad_row), B, K, V, r, _ptr(tokens), _ptr(logits),
        _ptr(draft_probs), _ptr(workspace.buffer), workspace.nbytes,
        _stream(stream))
    _lib.check("dspark_draft_block", st)
    return tokens, logits, draft_probs


def draft_block_per_request(base_logits, U, Wb, d0, seed, offset, temperature, *,
                            greedy=None, pad_row=None, tokens=None, logits=None,
                            draft_probs=None, slot=None,
                            workspace: Optional[DraftWorkspace] = None,
                            stream=None):
    """draft_block with temperature [B] float32 (device) per request and,
    when slot [B] int32 is given, proposals written to draft_probs[slot[b]]
    (draft_probs [num_slots, K, V], which must then be passed in).  Returns
    (tokens, logits, draft_probs).  See include/dspark.h."""
    torch = _torch()
    B, K, V = base_logits.shape
    r = U.shape[1]
    if tuple(U.shape) != (V, r) or tuple(Wb.shape) != (r, V):
        raise ValueError("U must be [V, r] and Wb [r, V]")
    if U.dtype != Wb.dtype:
        raise TypeError("U and Wb must share a dtype")
    if temperature.dtype != torch.float32 or tuple(temperature.shape) != (B,):
        raise TypeError("temperature must be float32 [B]")
    for t in (base_logits, U, Wb, d0, seed, offset, greedy, pad_row, temperature,
              slot):
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    dev = base_logits.device
    if slot is not None:
        if slot.dtype != torch.int32 or tuple(slot.shape) != (B,):
            raise TypeError("slot must be int32 [B]")
        if draft_probs is None or draft_probs.dim() != 3 or \
                tuple(draft_probs.shape[1:]) != (K, V):
            raise ValueError("with slot, pass draft_probs [num_slots, K, V]")
        num_slots = draft_probs.shape[0]
    else:
        num_slots = 0
    if tokens is None:
        tokens = torch.empty((B, K), dtype=torch.int32, device=dev)
    if logits is None:
        logits = torch.empty((B, K, V), dtype=torch.float32, device=dev)
    if draft_probs is None:
        draft_probs = torch.empty((B, K, V), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = DraftWorkspace(B, K, V, r, device=dev)
    st = _lib.load().dspark_draft_block_per_request(
        _ptr(base_logits), _dtype_code(base_logits), _ptr(U), _ptr(Wb),
        _dtype_code(U), _ptr(d0), _ptr(seed), _ptr(offset), _ptr(temperature),
        _ptr(greedy), _ptr(pad_row), B, K, V, r, _ptr(tokens), _ptr(logits),
        _ptr(draft_probs), _ptr(slot), num_slots, _ptr(workspace.buffer),
        workspace.nbytes, _stream(stream))
    _lib.check("dspark_draft_block_per_request", st)
    return tokens, logits, draft_probs


class HostWorkspace:
    """Device scratch for dspark_draft_block_host, sized for (B, K, V, r)."""

    def __init__(self, B: int, K: int, V: int, r: int, device=None):
        torch = _torch()
        n = int(_lib.load().dspark_draft_host_workspace_bytes(B, K, V, r))
        if n == 0:
            raise DsparkError("dspark_draft_host_workspace_bytes", 2)
        self.nbytes = n
        self.buffer = torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def draft_block_host(base_logits_host, U, Wb, d0_host, seed_host,
                     offset_host, T: float, *, base_dev, logits, draft_probs,
                     tokens_host=None, greedy_host=None, pad_row_host=None,
                     workspace: Optional[HostWorkspace] = None, stream=None,
                     copy_stream=None):
    """dspark_draft_block_host: inputs in (pinned) host tensors, tokens back
    to a host tensor; base_dev [B,K,V] receives the drafter logits on the
    device, copied position by position on ``copy_stream`` while earlier
    positions compute on ``stream``.  Returns tokens_host."""
    torch = _torch()
    B, K, V = base_logits_host.shape
    r = U.shape[1]
    if base_logits_host.is_cuda or d0_host.is_cuda:
        raise ValueError("base_logits_host and the per-request inputs must "
                         "be host tensors")
    if tuple(base_dev.shape) != (B, K, V) or base_dev.dtype != base_logits_host.dtype:
        raise ValueError("base_dev must match base_logits_host")
    if tokens_host is None:
        tokens_host = torch.empty((B, K), dtype=torch.int32).pin_memory()
    if workspace is None:
        workspace = HostWorkspace(B, K, V, r, device=base_dev.device)
    if copy_stream is None:
        raise ValueError("copy_stream is required (a stream other than stream)")
    st = _lib.load().dspark_draft_block_host(
        _ptr(base_logits_host), _dtype_code(base_logits_host), _ptr(U),
        _ptr(Wb), _dtype_code(U), _ptr(d0_host), _ptr(seed_host),
        _ptr(offset_host), float(T), _ptr(greedy_host), _ptr(pad_row_host),
        B, K, V, r, _ptr(base_dev), _ptr(tokens_host), _ptr(logits),
        _ptr(draft_probs), _ptr(workspace.buffer), workspace.nbytes,
        _stream(stream), copy_stream.cuda_stream)
    _lib.check("dspark_draft_block_host", st)
    return tokens_host


def draft_block_noalloc(base_logits, U, Wb, d0, seed, offset, T: float, *,
                        greedy=None, pad_row=None, tokens=None, logits=None,
                        draft_probs=None, stream=None):
    """dspark_draft_block_noalloc: the draft block with library-owned scratch
    instead of a caller-provided workspace, for callers that cannot allocate
    device memory.  The library call itself allocates nothing.  Outputs that
    are not passed in are allocated here by torch, for convenience; a caller
    that must not allocate passes tokens, logits and draft_probs.  Returns
    (tokens, logits, draft_probs)."""
    torch = _torch()
    B, K, V, r = _check_draft_inputs(base_logits, U, Wb, d0, seed, offset,
                                     greedy, pad_row, tokens, logits,
                                     draft_probs)
    dev = base_logits.device
    if tokens is None:
        tokens = torch.empty((B, K), dtype=torch.int32, device=dev)
    if logits is None:
        logits = torch.empty((B, K, V), dtype=torch.float32, device=dev)
    if draft_probs is None:
        draft_probs = torch.empty((B, K, V), dtype=torch.float32, device=dev)
    st = _lib.load().dspark_draft_block_noalloc(
        _ptr(base_logits), _dtype_code(base_logits), _ptr(U), _ptr(Wb),
        _dtype_code(U), _ptr(d0), _ptr(seed), _ptr(offset), float(T),
        _ptr(greedy), _ptr(pad_row), B, K, V, r, _ptr(tokens), _ptr(logits),
        _ptr(draft_probs), _stream(stream))
    _lib.check("dspark_draft_block_noalloc", st)
    return tokens, logits, draft_probs


def draft_block_profile(base_logits, U, Wb, d0, seed, offset, T: float, *,
                        greedy=None, pad_row=None, tokens=None, logits=None,
                        draft_probs=None, workspace=None, stream=None):
    """dspark_draft_block_profile: runs one block with CUDA events around
    every launch and returns {class: (total_ms, launches)} for the classes
    "position", "pick" and "proposal" (synchronises; not capturable)."""
    torch = _torch()
    B, K, V, r = _check_draft_inputs(base_logits, U, Wb, d0, seed, offset,
                                     greedy, pad_row, tokens, logits,
                                     draft_probs)
    dev = base_logits.device
    if tokens is None:
        tokens = torch.empty((B, K), dtype=torch.int32, device=dev)
    if logits is None:
        logits = torch.empty((B, K, V), dtype=torch.float32, device=dev)
    if draft_probs is None:
        draft_probs = torch.empty((B, K, V), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = DraftWorkspace(B, K, V, r, device=dev)
    ms = (ctypes.c_float * 3)()
    n = (ctypes.c_int * 3)()
    st = _lib.load().dspark_draft_block_profile(
        _ptr(base_logits), _dtype_code(base_logits), _ptr(U), _ptr(Wb),
        _dtype_code(U), _ptr(d0), _ptr(seed), _ptr(offset), float(T),
        _ptr(greedy), _ptr(pad_row), B, K, V, r, _ptr(tokens), _ptr(logits),
        _ptr(draft_probs), _ptr(workspace.buffer), workspace.nbytes,
        ctypes.cast(ms, ctypes.c_void_p), ctypes.cast(n, ctypes.c_void_p),
        _stream(stream))
    _lib.check("dspark_draft_block_profile", st)
    names = ("position", "pick", "proposal")
    return {names[i]: (float(ms[i]), int(n[i])) for i in range(3)}


def draft_block_timeline(base_logits, U, Wb, d0, seed, offset, T: float, *,
                         replays: int, stream, greedy=None, pad_row=None,
                         tokens=None, logits=None, draft_probs=None,
                         workspace=None):
    """dspark_draft_block_timeline: the block captured into a CUDA graph with
    event nodes around the position chain and the proposal writer, replayed
    ``replays`` times on ``stream`` (a created stream, not the default one).
    Returns (chain_ms, proposal_ms), the mean per replay (synchronises)."""
    torch = _torch()
    B, K, V, r = _check_draft_inputs(base_logits, U, Wb, d0, seed, offset,
                                     greedy, pad_row, tokens, logits,
                                     draft_probs)
    dev = base_logits.device
    if tokens is None:
        tokens = torch.empty((B, K), dtype=torch.int32, device=dev)
    if logits is None:
        logits = torch.empty((B, K, V), dtype=torch.float32, device=dev)
    if draft_probs is None:
        draft_probs = torch.empty((B, K, V), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = DraftWorkspace(B, K, V, r, device=dev)
    chain = ctypes.c_float(0.0)
    prop = ctypes.c_float(0.0)
    st = _lib.load().dspark_draft_block_timeline(
        _ptr(base_logits), _dtype_code(base_logits), _ptr(U), _ptr(Wb),
        _dtype_code(U), _ptr(d0), _ptr(seed), _ptr(offset), float(T),
        _ptr(greedy), _ptr(pad_row), B, K, V, r, _ptr(tokens), _ptr(logits),
        _ptr(draft_probs), _ptr(workspace.buffer), workspace.nbytes,
        int(replays), ctypes.byref(chain), ctypes.byref(prop),
        _stream(stream))
    _lib.check("dspark_draft_block_timeline", st)
    return float(chain.value), float(prop.value)


def _verify(fn, draft_probs, target_probs, tokens, seed, offset,
            accepted_len, emitted_token, stream):
    torch = _torch()
    B, K, V = draft_probs.shape
    if tuple(target_probs.shape) != (B, K + 1, V):
        raise ValueError("target_probs must be [B, K+1, V]")
    dev = draft_probs.device
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
    if emitted_token is None:
        emitted_token = torch.empty(B, dtype=torch.int32, device=dev)
    st = getattr(_lib.load(), fn)(
        _ptr(draft_probs), _ptr(target_probs), _ptr(tokens), _ptr(seed),
        _ptr(offset), B, K, V, _ptr(accepted_len), _ptr(emitted_token),
        _stream(stream))
    _lib.check(fn, st)
    return accepted_len, emitted_token


def verify_standard(draft_probs, target_probs, tokens, seed, offset, *,
                    accepted_len=None, emitted_token=None, stream=None):
    """Standard rejection verification.  Returns (accepted_len, emitted)."""
    return _verify("dspark_verify_standard", draft_probs, target_probs, tokens,
                   seed, offset, accepted_len, emitted_token, stream)


def verify_block(draft_probs, target_probs, tokens, seed, offset, *,
                 accepted_len=None, emitted_token=None, stream=None):
    """Block verification (same arguments and outputs as verify_standard).
    Returns (accepted_len, emitted)."""
    return _verify("dspark_verify_block", draft_probs, target_probs, tokens,
                   seed, offset, accepted_len, emitted_token, stream)


def sample_temperature(logits, seed, offset, *, T: float = 1.0,
                       temperature=None, greedy=None, position=None,
                       tokens=None, probs=None, with_probs: bool = True,
                       workspace=None, stream=None):
    """Temperature-only sampling of target rows: logits [R, V] float32 on
    the device, seed/offset [R] int64 (uint64 bit patterns), T (or
    temperature [R] float32), greedy [R] uint8, position [R] int32.  Returns
    (tokens [R], probs [R, V] or None).  See include/dspark.h."""
    torch = _torch()
    R, V = logits.shape
    for t in (logits, seed, offset, temperature, greedy, position):
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    dev = logits.device
    if tokens is None:
        tokens = torch.empty(R, dtype=torch.int32, device=dev)
    if with_probs and probs is None:
        probs = torch.empty((R, V), dtype=torch.float32, device=dev)
    if not with_probs:
        probs = None
    nbytes = _lib.load().dspark_sample_workspace_bytes(R, V)
    if nbytes == 0:
        raise _lib.DsparkError("dspark_sample_workspace_bytes", 2)
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = _lib.load().dspark_sample_temperature(
        _ptr(logits), _ptr(temperature), float(T), _ptr(greedy), _ptr(seed),
        _ptr(offset), _ptr(position), R, V, _ptr(tokens), _ptr(probs),
        _ptr(workspace), workspace.numel(), _stream(stream))
    _lib.check("dspark_sample_temperature", st)
    return tokens, probs


def noise_words(seed: int, offset: int, k: int, stream_id: int, n: int,
                device=None, with_gumbel: bool = True, stream=None,
                folded: bool = False):
    """Diagnostic: the raw Philox words (and float32 Gumbel variates) the
    kernels use for elements 0..n-1.  folded=True computes them the way the
    hot kernels do (dspark_noise_words_folded).  Returns (words int32-view,
    gumbel)."""
    torch = _torch()
    dev = device or "cuda"
    out = torch.empty(n, dtype=torch.int32, device=dev)
    g = torch.empty(n, dtype=torch.float32, device=dev) if with_gumbel else None
    fn = "dspark_noise_words_folded" if folded else "dspark_noise_words"
    st = getattr(_lib.load(), fn)(seed, offset, k, stream_id, n, _ptr(out),
                                  _ptr(g), _stream(stream))
    _lib.check(fn, st)
    return out, g


def read_device_error(workspace: DraftWorkspace, stream=None) -> int:
    """Reads and clears the workspace's device error word (synchronises)."""
    code = ctypes.c_int(0)
    st = _lib.load().dspark_read_device_error(
        _ptr(workspace.buffer), ctypes.byref(code), _stream(stream))
    if st not in (0, 5):
        _lib.check("dspark_read_device_error", st)
    return code.value
