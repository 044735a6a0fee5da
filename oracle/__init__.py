"""CPU oracle for DSpark ancestral draft-block sampling -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` legs may import this package.  The
product path (``ancestral_draft_sampling_gb300``) never imports it and shares
no code with it.

The arithmetic lives in ``dspark_oracle.c`` (plain C, double accumulation);
this module only compiles it with gcc and marshals numpy arrays through
ctypes.  Every function cites the passage of the pages it follows in the C
file's comments.

Parity status: every oracle function is pinned by ``tests/test_oracle_pins.py``
(Philox known answers and cuRAND's host generator, the Gumbel CDF, chi-square
of Gumbel-max against the closed-form softmax, conditioning, the greedy chain
against numpy's argmax, the bias against a float64 GEMV, proposal sums, and
losslessness of standard verification) and ``tests/test_oracle_block.py``
(block verification: losslessness by chi-square, its reduction to the
standard rule at K = 1, identical draft and target) and
``tests/test_oracle_sampler.py`` (temperature-only sampling: chi-square
against the closed-form softmax, the draft positions' softmax, greedy rows,
independent noise streams).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to the source (gcc, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11",
           "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        U64 = ctypes.c_uint64
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_noise_word.argtypes = [U64, U64, I, I, ctypes.c_uint32]
        lib.oracle_noise_word.restype = ctypes.c_uint32
        lib.oracle_noise_words.argtypes = [U64, U64, I, I, ctypes.c_uint32, P]
        lib.oracle_noise_words.restype = None
        lib.oracle_gumbel.argtypes = [ctypes.c_uint32]
        lib.oracle_gumbel.restype = ctypes.c_double
        lib.oracle_accept_uniform.argtypes = [ctypes.c_uint32]
        lib.oracle_accept_uniform.restype = ctypes.c_float
        lib.oracle_draft_position.argtypes = [
            P, I, I, P, P, I, I, I, I, U64, U64, I, ctypes.c_float, I,
            P, P, P, P, P, P, P, P]
        lib.oracle_draft_position.restype = I
        lib.oracle_draft_block.argtypes = [
            P, I, P, P, I, P, P, P, ctypes.c_float, P, P, I, I, I, I,
            P, P, P, P, P, P]
        lib.oracle_draft_block.restype = I
        lib.oracle_verify_standard.argtypes = [P, P, P, P, P, I, I, I, P, P,
                                               P, P]
        lib.oracle_verify_standard.restype = I
        lib.oracle_verify_block.argtypes = [P, P, P, P, P, I, I, I, P, P, P, P,
                                            P, P]
        lib.oracle_verify_block.restype = I
        lib.oracle_sample_temperature.argtypes = [P, P, P, P, P, P, I, I, P, P,
                                                  P, P, P]
        lib.oracle_sample_temperature.restype = I
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:  # bfloat16 bit patterns
        return BF16
    raise TypeError(f"oracle takes float32 or bf16 bits (uint16), got {a.dtype}")


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def noise_word(seed: int, offset: int, k: int, stream: int, index: int) -> int:
    return int(_load().oracle_noise_word(seed, offset, k, stream, index))


def noise_words(seed: int, offset: int, k: int, stream: int, n: int) -> np.ndarray:
    """Words of elements 0 .. n-1: ``noise_word`` for each index."""
    out = np.empty(n, dtype=np.uint32)
    _load().oracle_noise_words(seed, offset, k, stream, n, _ptr(out))
    return out


def gumbel(x: int) -> float:
    return float(_load().oracle_gumbel(x))


def accept_uniform(x: int) -> float:
    return float(_load().oracle_accept_uniform(x))


class PositionResult:
    __slots__ = ("logits", "probs", "token", "M", "S", "best", "second")


def draft_position(base_row, U, Wb, prev, seed, offset, k, T, greedy=False,
                   is_pad=False) -> PositionResult:
    """One (request, position): see ``oracle_draft_position`` in the C file."""
    lib = _load()
    V, r = U.shape
    assert Wb.shape == (r, V) and U.dtype == Wb.dtype
    w_dtype = _dtype_code(U)
    if base_row is None:
        base_row_c, base_dtype = None, F32
        assert is_pad
    else:
        base_row_c = np.ascontiguousarray(base_row)
        base_dtype = _dtype_code(base_row_c)
    U = np.ascontiguousarray(U)
    Wb = np.ascontiguousarray(Wb)
    res = PositionResult()
    res.logits = np.empty(V, dtype=np.float32)
    res.probs = np.empty(V, dtype=np.float64)
    tok = np.zeros(1, dtype=np.int32)
    M = np.zeros(1, dtype=np.float64)
    S = np.zeros(1, dtype=np.float64)
    best = np.zeros(1, dtype=np.float32)
    second = np.zeros(1, dtype=np.float32)
    scratch = np.empty(V, dtype=np.float64)
    rc = lib.oracle_draft_position(
        _ptr(base_row_c), base_dtype, int(bool(is_pad)), _ptr(U), _ptr(Wb),
        w_dtype, V, r, int(prev), int(seed), int(offset), int(k), float(T),
        int(bool(greedy)), _ptr(res.logits), _ptr(res.probs), _ptr(tok),
        _ptr(M), _ptr(S), _ptr(best), _ptr(second), _ptr(scratch))
    if rc != 0:
        raise ValueError("oracle_draft_position rejected its arguments")
    res.token = int(tok[0])
    res.M = float(M[0])
    res.S = float(S[0])
    res.best = float(best[0])
    res.second = float(second[0])
    return res


class BlockResult:
    __slots__ = ("tokens", "logits", "probs", "rowstats", "top2")


def request_temperatures(T, B):
    """Per-request temperatures from a scalar or a [B] array; a value that is
    not finite and positive counts as 1 (the per-request entry point's
    reading)."""
    if np.ndim(T) == 0:
        return np.full(B, float(T), dtype=np.float32)
    t = np.asarray(T, dtype=np.float32).copy()
    t[~(np.isfinite(t) & (t > 0))] = 1.0
    return t


def draft_block(base, U, Wb, d0, seed, offset, T, greedy=None,
                pad_row=None) -> BlockResult:
    """The whole ancestral block, row after row (single thread).  T is a
    scalar, or a [B] array of per-request temperatures (then each request
    runs as its own block with its own T)."""
    if np.ndim(T) > 0:
        B = base.shape[0]
        Ts = request_temperatures(T, B)
        parts = [draft_block(base[b:b + 1], U, Wb, d0[b:b + 1], seed[b:b + 1],
                             offset[b:b + 1], float(Ts[b]),
                             None if greedy is None else greedy[b:b + 1],
                             None if pad_row is None else pad_row[b:b + 1])
                 for b in range(B)]
        out = BlockResult()
        for name in BlockResult.__slots__:
            setattr(out, name, np.concatenate([getattr(x, name) for x in parts]))
        return out
    lib = _load()
    B, K, V = base.shape
    r = U.shape[1]
    base = np.ascontiguousarray(base)
    U = np.ascontiguousarray(U)
    Wb = np.ascontiguousarray(Wb)
    d0 = np.ascontiguousarray(d0, dtype=np.int32)
    seed = np.ascontiguousarray(seed, dtype=np.uint64)
    offset = np.ascontiguousarray(offset, dtype=np.uint64)
    g = None if greedy is None else np.ascontiguousarray(greedy, dtype=np.uint8)
    p = None if pad_row is None else np.ascontiguousarray(pad_row, dtype=np.uint8)
    out = BlockResult()
    out.tokens = np.zeros((B, K), dtype=np.int32)
    out.logits = np.empty((B, K, V), dtype=np.float32)
    out.probs = np.empty((B, K, V), dtype=np.float64)
    out.rowstats = np.empty((B, K, 2), dtype=np.float64)
    out.top2 = np.empty((B, K, 2), dtype=np.float32)
    scratch = np.empty(V, dtype=np.float64)
    rc = lib.oracle_draft_block(
        _ptr(base), _dtype_code(base), _ptr(U), _ptr(Wb), _dtype_code(U),
        _ptr(d0), _ptr(seed), _ptr(offset), float(T), _ptr(g), _ptr(p), B, K,
        V, r, _ptr(out.tokens), _ptr(out.logits), _ptr(out.probs),
        _ptr(out.rowstats), _ptr(out.top2), _ptr(scratch))
    if rc != 0:
        raise ValueError("oracle_draft_block rejected its arguments")
    return out


def draft_chains(base, U, Wb, d0, seed, offset, T, depth, greedy=None,
                 pad_row=None, threads: int | None = None):
    """Free-running chains: for each request b with depth[b] > 0, positions
    0 .. depth[b]-1 in order, each conditioned on the oracle's own draw
    before it (d0[b] for position 0), exactly as ``draft_block`` computes
    them.  Requests are independent, so they run on a thread pool (ctypes
    releases the GIL).  Returns {b: [PositionResult per position]}."""
    todo = [b for b in range(len(depth)) if depth[b] > 0]
    threads = threads or max(1, min(len(todo), os.cpu_count() or 1))
    Ts = request_temperatures(T, len(depth))  # T: scalar or per request

    def one(b):
        is_pad = bool(pad_row[b]) if pad_row is not None else False
        is_greedy = bool(greedy[b]) if greedy is not None else False
        prev, chain = int(d0[b]), []
        for k in range(int(depth[b])):
            row = None if is_pad else base[b, k]
            res = draft_position(row, U, Wb, prev, int(seed[b]),
                                 int(offset[b]), k, float(Ts[b]),
                                 greedy=is_greedy, is_pad=is_pad)
            chain.append(res)
            prev = res.token
        return chain

    if not todo:
        return {}
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return dict(zip(todo, ex.map(one, todo)))


class VerifyResult:
    __slots__ = ("accepted_len", "emitted", "top2", "h", "eta")


def verify_standard(draft_probs, target_probs, tokens, seed, offset) -> VerifyResult:
    lib = _load()
    B, K, V = draft_probs.shape
    assert target_probs.shape == (B, K + 1, V)
    q = np.ascontiguousarray(draft_probs, dtype=np.float32)
    p = np.ascontiguousarray(target_probs, dtype=np.float32)
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    s = np.ascontiguousarray(seed, dtype=np.uint64)
    o = np.ascontiguousarray(offset, dtype=np.uint64)
    out = VerifyResult()
    out.accepted_len = np.zeros(B, dtype=np.int32)
    out.emitted = np.zeros(B, dtype=np.int32)
    out.top2 = np.zeros((B, 2), dtype=np.float32)
    scratch = np.empty(V, dtype=np.float32)
    rc = lib.oracle_verify_standard(_ptr(q), _ptr(p), _ptr(t), _ptr(s), _ptr(o),
                                    B, K, V, _ptr(out.accepted_len),
                                    _ptr(out.emitted), _ptr(out.top2),
                                    _ptr(scratch))
    if rc != 0:
        raise ValueError("oracle_verify_standard rejected its arguments")
    return out


def verify_block(draft_probs, target_probs, tokens, seed, offset) -> VerifyResult:
    """Block verification (PR #21, "2. Golden sampling semantics": the
    ``block`` rejection_sample_method, Sun et al. 2024), see
    oracle_verify_block.  Besides accepted_len, emitted and top2 the result
    holds ``h`` [B,K] (float64: the thresholds h_1..h_K) and ``eta`` [B,K]
    (float32: the uniforms they are compared with)."""
    lib = _load()
    B, K, V = draft_probs.shape
    assert target_probs.shape == (B, K + 1, V)
    q = np.ascontiguousarray(draft_probs, dtype=np.float32)
    p = np.ascontiguousarray(target_probs, dtype=np.float32)
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    s = np.ascontiguousarray(seed, dtype=np.uint64)
    o = np.ascontiguousarray(offset, dtype=np.uint64)
    out = VerifyResult()
    out.accepted_len = np.zeros(B, dtype=np.int32)
    out.emitted = np.zeros(B, dtype=np.int32)
    out.top2 = np.zeros((B, 2), dtype=np.float32)
    out.h = np.zeros((B, K), dtype=np.float64)
    out.eta = np.zeros((B, K), dtype=np.float32)
    scratch = np.empty(V, dtype=np.float32)
    rc = lib.oracle_verify_block(_ptr(q), _ptr(p), _ptr(t), _ptr(s), _ptr(o),
                                 B, K, V, _ptr(out.accepted_len),
                                 _ptr(out.emitted), _ptr(out.top2),
                                 _ptr(out.h), _ptr(out.eta), _ptr(scratch))
    if rc != 0:
        raise ValueError("oracle_verify_block rejected its arguments")
    return out


class SampleResult:
    __slots__ = ("tokens", "probs", "rowstats", "top2")


def sample_temperature(logits, T, seed, offset, greedy=None,
                       position=None) -> SampleResult:
    """Temperature-only target sampling (PR #27, "1. Temperature-only
    sampling runs no filter"), see oracle_sample_temperature.  logits [R,V]
    float32; T scalar or [R] (an invalid value counts as 1, the reading of
    the per-request entry points)."""
    lib = _load()
    R, V = logits.shape
    x = np.ascontiguousarray(logits, dtype=np.float32)
    t = request_temperatures(T, R)
    s = np.ascontiguousarray(seed, dtype=np.uint64)
    o = np.ascontiguousarray(offset, dtype=np.uint64)
    g = None if greedy is None else np.ascontiguousarray(greedy, dtype=np.uint8)
    pos = None if position is None else np.ascontiguousarray(position, dtype=np.int32)
    out = SampleResult()
    out.tokens = np.zeros(R, dtype=np.int32)
    out.probs = np.empty((R, V), dtype=np.float64)
    out.rowstats = np.empty((R, 2), dtype=np.float64)
    out.top2 = np.empty((R, 2), dtype=np.float32)
    scratch = np.empty(V, dtype=np.float64)
    rc = lib.oracle_sample_temperature(
        _ptr(x), _ptr(t), _ptr(g), _ptr(s), _ptr(o), _ptr(pos), R, V,
        _ptr(out.tokens), _ptr(out.probs), _ptr(out.rowstats), _ptr(out.top2),
        _ptr(scratch))
    if rc != 0:
        raise ValueError("oracle_sample_temperature rejected its arguments")
    return out
