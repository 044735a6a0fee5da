"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, sizes its workspace, and rejects bad arguments with a status
before any launch.  Every call here fails a host-side check, so no kernel is
ever launched (the fake device addresses are never dereferenced)."""
import os
import re

import pytest

from ancestral_draft_sampling_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")

FAKE = 0x7F0000000000  # 256-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DSPARK_API\s+[\w\s\*]+?\b(dspark_\w+)\s*\(", text)))


def test_header_declares_the_binding_list():
    assert declared_symbols() == sorted(_lib.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert lib.dspark_version().decode().count(".") == 2


def test_status_strings(lib):
    for code, name in _lib.STATUS.items():
        assert lib.dspark_status_string(code).decode() == name
    assert lib.dspark_status_string(99).decode() == "DSPARK_UNKNOWN_STATUS"


def test_workspace_bytes(lib):
    ws = lib.dspark_draft_workspace_bytes
    assert ws(88, 7, 200064, 256) > 0
    assert ws(88, 7, 200064, 256) >= ws(8, 7, 200064, 256)
    assert ws(1, 3, 4096, 64) % 256 == 0
    for bad in [(0, 7, 100, 64), (8, 0, 100, 64), (8, 7, 0, 64),
                (8, 7, 100, 8), (8, 7, 100, 72), (8, 7, 100, 512),
                (2000, 7, 100, 64), (8, 100, 100, 64), (8, 7, (1 << 26) + 1, 64)]:
        assert ws(*bad) == 0, bad


def _draft_args(lib, **over):
    B, K, V, r = 4, 3, 1024, 64
    a = dict(base=FAKE, base_dtype=0, U=FAKE, Wb=FAKE, w_dtype=1, d0=FAKE,
             seed=FAKE, offset=FAKE, T=1.0, greedy=None, pad_row=None, B=B,
             K=K, V=V, r=r, tokens=FAKE, logits=FAKE, probs=FAKE,
             workspace=FAKE, ws_bytes=lib.dspark_draft_workspace_bytes(B, K, V, r),
             stream=None)
    a.update(over)
    return a


def _call(lib, a):
    return lib.dspark_draft_block(
        a["base"], a["base_dtype"], a["U"], a["Wb"], a["w_dtype"], a["d0"],
        a["seed"], a["offset"], a["T"], a["greedy"], a["pad_row"], a["B"],
        a["K"], a["V"], a["r"], a["tokens"], a["logits"], a["probs"],
        a["workspace"], a["ws_bytes"], a["stream"])


INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 3


@pytest.mark.parametrize("over,want", [
    (dict(base=None), INVALID),
    (dict(U=None), INVALID),
    (dict(Wb=None), INVALID),
    (dict(d0=None), INVALID),
    (dict(seed=None), INVALID),
    (dict(offset=None), INVALID),
    (dict(tokens=None), INVALID),
    (dict(logits=None), INVALID),
    (dict(probs=None), INVALID),
    (dict(T=0.0), INVALID),
    (dict(T=-1.0), INVALID),
    (dict(T=float("nan")), INVALID),
    (dict(T=float("inf")), INVALID),
    (dict(base_dtype=2), INVALID),
    (dict(w_dtype=7), INVALID),
    (dict(B=0), INVALID),
    (dict(K=0), INVALID),
    (dict(V=-5), INVALID),
    (dict(base=FAKE + 4), INVALID),
    (dict(logits=FAKE + 8), INVALID),
    (dict(greedy=FAKE + 1), INVALID),
    (dict(r=40), UNSUPPORTED),
    (dict(r=512), UNSUPPORTED),
    (dict(B=5000), UNSUPPORTED),
    (dict(K=65), UNSUPPORTED),
    (dict(workspace=None), WORKSPACE),
    (dict(ws_bytes=100), WORKSPACE),
    (dict(workspace=FAKE + 16), WORKSPACE),
])
def test_draft_block_rejects_bad_arguments(lib, over, want):
    assert _call(lib, _draft_args(lib, **over)) == want


def test_verify_rejects_bad_arguments(lib):
    f = lib.dspark_verify_standard
    good = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, 3, 100, FAKE, FAKE, None]
    for i in [0, 1, 2, 3, 4, 8, 9]:
        args = list(good)
        args[i] = None
        assert f(*args) == INVALID
    for i, v in [(5, 0), (6, 0), (7, 0)]:
        args = list(good)
        args[i] = v
        assert f(*args) == INVALID
    args = list(good)
    args[0] = FAKE + 4
    assert f(*args) == INVALID
    args = list(good)
    args[6] = 65
    assert f(*args) == UNSUPPORTED


def test_noise_words_rejects_bad_arguments(lib):
    f = lib.dspark_noise_words
    assert f(1, 2, 0, 0, 0, FAKE, None, None) == INVALID
    assert f(1, 2, 0, 0, 16, None, None, None) == INVALID
    assert f(1, 2, -1, 0, 16, FAKE, None, None) == INVALID
    assert f(1, 2, 0, 1 << 17, 16, FAKE, None, None) == INVALID
    assert f(1, 2, 0, 0, 16, FAKE + 4, None, None) == INVALID


def test_noise_words_folded_rejects_bad_arguments(lib):
    f = lib.dspark_noise_words_folded
    assert f(1, 2, 0, 0, 0, FAKE, None, None) == INVALID
    assert f(1, 2, 0, 0, 16, None, None, None) == INVALID
    assert f(1, 2, 0x10000, 0, 16, FAKE, None, None) == INVALID
    assert f(1, 2, 0, 0, 16, FAKE, FAKE + 8, None) == INVALID


def _timeline_call(lib, a, replays=3, chain=True, prop=True, stream=1):
    import ctypes
    c, p = ctypes.c_float(0), ctypes.c_float(0)
    return lib.dspark_draft_block_timeline(
        a["base"], a["base_dtype"], a["U"], a["Wb"], a["w_dtype"], a["d0"],
        a["seed"], a["offset"], a["T"], a["greedy"], a["pad_row"], a["B"],
        a["K"], a["V"], a["r"], a["tokens"], a["logits"], a["probs"],
        a["workspace"], a["ws_bytes"], replays,
        ctypes.byref(c) if chain else None, ctypes.byref(p) if prop else None,
        stream)


@pytest.mark.parametrize("kw,over,want", [
    (dict(stream=None), {}, INVALID),       # the legacy stream cannot capture
    (dict(replays=0), {}, INVALID),
    (dict(chain=False), {}, INVALID),
    (dict(prop=False), {}, INVALID),
    (dict(), dict(T=0.0), INVALID),         # the block's own checks
    (dict(), dict(r=40), UNSUPPORTED),
    (dict(), dict(ws_bytes=100), WORKSPACE),
])
def test_draft_block_timeline_rejects_bad_arguments(lib, kw, over, want):
    assert _timeline_call(lib, _draft_args(lib, **over), **kw) == want


def test_workspace_starts_with_the_error_word_row(lib):
    """The error word sits at offset 0 and the decision-key rows follow it
    at a 4 KB pitch, so one 2-D memset clears both: the workspace grows by
    one 4 KB row per request plus one for the error word."""
    ws = lib.dspark_draft_workspace_bytes
    per_request = ws(9, 7, 200064, 256) - ws(8, 7, 200064, 256)
    assert per_request >= 4096 + 2 * 512 * 16
    assert ws(1, 1, 16, 16) >= 2 * 4096


def test_read_device_error_rejects_null(lib):
    import ctypes
    code = ctypes.c_int(0)
    assert lib.dspark_read_device_error(None, ctypes.byref(code), None) == INVALID
    assert lib.dspark_read_device_error(FAKE, None, None) == INVALID


def test_host_workspace_bytes(lib):
    wh = lib.dspark_draft_host_workspace_bytes
    ws = lib.dspark_draft_workspace_bytes
    assert wh(88, 7, 200064, 256) > ws(88, 7, 200064, 256)
    assert wh(88, 7, 200064, 256) % 256 == 0
    assert wh(0, 7, 100, 64) == 0


def _host_args(lib, **over):
    import ctypes
    B, K, V, r = 4, 3, 1024, 64
    host = (ctypes.c_uint8 * 64)()  # host stand-in, never read: every call fails first
    h = ctypes.addressof(host)
    a = dict(base=h, base_dtype=0, U=FAKE, Wb=FAKE, w_dtype=1, d0=h, seed=h,
             offset=h, T=1.0, greedy=None, pad_row=None, B=B, K=K, V=V, r=r,
             base_dev=FAKE, tokens=h, logits=FAKE, probs=FAKE, ws=FAKE,
             ws_bytes=lib.dspark_draft_host_workspace_bytes(B, K, V, r),
             stream=None, copy_stream=1)
    a.update(over)
    return host, a


@pytest.mark.parametrize("over,want", [
    (dict(base=None), 1), (dict(d0=None), 1), (dict(tokens=None), 1),
    (dict(base_dev=None), 1), (dict(copy_stream=None), 1),   # same as stream
    (dict(T=0.0), 1), (dict(base_dev=FAKE + 8), 1), (dict(r=72), 2),
    (dict(ws=None), 3), (dict(ws_bytes=256), 3), (dict(ws=FAKE + 16), 3),
])
def test_draft_block_host_rejects_bad_arguments(lib, over, want):
    host, a = _host_args(lib, **over)
    st = lib.dspark_draft_block_host(
        a["base"], a["base_dtype"], a["U"], a["Wb"], a["w_dtype"], a["d0"],
        a["seed"], a["offset"], a["T"], a["greedy"], a["pad_row"], a["B"],
        a["K"], a["V"], a["r"], a["base_dev"], a["tokens"], a["logits"],
        a["probs"], a["ws"], a["ws_bytes"], a["stream"], a["copy_stream"])
    assert st == want


def test_verify_block_rejects_bad_arguments(lib):
    f = lib.dspark_verify_block
    good = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, 3, 100, FAKE, FAKE, None]
    for i in [0, 1, 2, 3, 4, 8, 9]:
        args = list(good)
        args[i] = None
        assert f(*args) == INVALID
    for i, v in [(5, 0), (6, 0), (7, 0)]:
        args = list(good)
        args[i] = v
        assert f(*args) == INVALID
    args = list(good)
    args[1] = FAKE + 8
    assert f(*args) == INVALID
    args = list(good)
    args[6] = 65
    assert f(*args) == UNSUPPORTED


def _per_request_call(lib, a, temperature=FAKE, slot=None, num_slots=0):
    return lib.dspark_draft_block_per_request(
        a["base"], a["base_dtype"], a["U"], a["Wb"], a["w_dtype"], a["d0"],
        a["seed"], a["offset"], temperature, a["greedy"], a["pad_row"], a["B"],
        a["K"], a["V"], a["r"], a["tokens"], a["logits"], a["probs"], slot,
        num_slots, a["workspace"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,over,want", [
    (dict(temperature=None), {}, INVALID),          # the per-request values
    (dict(temperature=FAKE + 2), {}, INVALID),      # 4-byte alignment
    (dict(slot=FAKE, num_slots=0), {}, INVALID),    # slots need num_slots
    (dict(slot=FAKE + 1, num_slots=8), {}, INVALID),
    (dict(), dict(base=None), INVALID),             # the block's own checks
    (dict(), dict(r=40), UNSUPPORTED),
    (dict(), dict(ws_bytes=100), WORKSPACE),
])
def test_draft_block_per_request_rejects_bad_arguments(lib, kw, over, want):
    assert _per_request_call(lib, _draft_args(lib, **over), **kw) == want


def test_sample_workspace_bytes(lib):
    f = lib.dspark_sample_workspace_bytes
    assert f(704, 200064) > 0 and f(704, 200064) % 256 == 0
    assert f(0, 100) == 0 and f(10, 0) == 0 and f(70000, 100) == 0


def _sample_call(lib, **over):
    R, V = 6, 1000
    a = dict(logits=FAKE, temperature=None, T=1.0, greedy=None, seed=FAKE,
             offset=FAKE, position=None, R=R, V=V, tokens=FAKE, probs=FAKE,
             ws=FAKE, ws_bytes=lib.dspark_sample_workspace_bytes(R, V),
             stream=None)
    a.update(over)
    return lib.dspark_sample_temperature(
        a["logits"], a["temperature"], a["T"], a["greedy"], a["seed"],
        a["offset"], a["position"], a["R"], a["V"], a["tokens"], a["probs"],
        a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,want", [
    (dict(logits=None), INVALID), (dict(seed=None), INVALID),
    (dict(tokens=None), INVALID), (dict(R=0), INVALID), (dict(V=0), INVALID),
    (dict(T=0.0), INVALID), (dict(T=float("nan")), INVALID),
    (dict(logits=FAKE + 4), INVALID), (dict(position=FAKE + 2), INVALID),
    (dict(temperature=FAKE + 1), INVALID),
    (dict(R=70000), UNSUPPORTED),
    (dict(ws=None), WORKSPACE), (dict(ws_bytes=64), WORKSPACE),
    (dict(ws=FAKE + 16), WORKSPACE),
])
def test_sample_temperature_rejects_bad_arguments(lib, over, want):
    assert _sample_call(lib, **over) == want
