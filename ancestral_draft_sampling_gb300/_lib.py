"""ctypes binding of libdspark.so (the C ABI in include/dspark.h).

Argument marshalling only: every step of the sampler runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams.  There is no CPU
fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdspark.so")

F32, BF16 = 0, 1

STATUS = {
    0: "DSPARK_OK",
    1: "DSPARK_ERR_INVALID_ARG",
    2: "DSPARK_ERR_UNSUPPORTED",
    3: "DSPARK_ERR_WORKSPACE",
    4: "DSPARK_ERR_CUDA",
    5: "DSPARK_ERR_DEVICE",
}

# Every symbol include/dspark.h declares.
EXPORTED = (
    "dspark_draft_workspace_bytes",
    "dspark_draft_block_per_request",
    "dspark_draft_block",
    "dspark_draft_block_profile",
    "dspark_draft_block_timeline",
    "dspark_draft_block_noalloc",
    "dspark_draft_host_workspace_bytes",
    "dspark_draft_block_host",
    "dspark_verify_standard",
    "dspark_sample_workspace_bytes",
    "dspark_sample_temperature",
    "dspark_verify_block",
    "dspark_noise_words",
    "dspark_noise_words_folded",
    "dspark_read_device_error",
    "dspark_status_string",
    "dspark_version",
)


class DsparkError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Loads the in-tree libdspark.so (built by __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
        lib.dspark_draft_workspace_bytes.argtypes = [I, I, I, I]
        lib.dspark_draft_workspace_bytes.restype = ctypes.c_size_t
        lib.dspark_draft_block.argtypes = [
            P, I, P, P, I, P, P, P, ctypes.c_float, P, P, I, I, I, I, P, P, P,
            P, ctypes.c_size_t, P]
        lib.dspark_draft_block.restype = I
        lib.dspark_draft_block_profile.argtypes = [
            P, I, P, P, I, P, P, P, ctypes.c_float, P, P, I, I, I, I, P, P, P,
            P, ctypes.c_size_t, P, P, P]
        lib.dspark_draft_block_profile.restype = I
        lib.dspark_draft_block_timeline.argtypes = [
            P, I, P, P, I, P, P, P, ctypes.c_float, P, P, I, I, I, I, P, P, P,
            P, ctypes.c_size_t, I, P, P, P]
        lib.dspark_draft_block_timeline.restype = I
        lib.dspark_draft_block_noalloc.argtypes = [
            P, I, P, P, I, P, P, P, ctypes.c_float, P, P, I, I, I, I, P, P, P,
            P]
        lib.dspark_draft_block_noalloc.restype = I
        lib.dspark_draft_host_workspace_bytes.argtypes = [I, I, I, I]
        lib.dspark_draft_host_workspace_bytes.restype = ctypes.c_size_t
        lib.dspark_draft_block_host.argtypes = [
            P, I, P, P, I, P, P, P, ctypes.c_float, P, P, I, I, I, I, P, P, P,
            P, P, ctypes.c_size_t, P, P]
        lib.dspark_draft_block_host.restype = I
        lib.dspark_verify_standard.argtypes = [P, P, P, P, P, I, I, I, P, P, P]
        lib.dspark_verify_standard.restype = I
        lib.dspark_verify_block.argtypes = [P, P, P, P, P, I, I, I, P, P, P]
        lib.dspark_verify_block.restype = I
        lib.dspark_draft_block_per_request.argtypes = [
            P, I, P, P, I, P, P, P, P, P, P, I, I, I, I, P, P, P, P, I, P,
            ctypes.c_size_t, P]
        lib.dspark_draft_block_per_request.restype = I
        lib.dspark_sample_workspace_bytes.argtypes = [I, I]
        lib.dspark_sample_workspace_bytes.restype = ctypes.c_size_t
        lib.dspark_sample_temperature.argtypes = [
            P, P, ctypes.c_float, P, P, P, P, I, I, P, P, P, ctypes.c_size_t, P]
        lib.dspark_sample_temperature.restype = I
        lib.dspark_noise_words.argtypes = [U64, U64, I, I, I, P, P, P]
        lib.dspark_noise_words.restype = I
        lib.dspark_noise_words_folded.argtypes = [U64, U64, I, I, I, P, P, P]
        lib.dspark_noise_words_folded.restype = I
        lib.dspark_read_device_error.argtypes = [P, P, P]
        lib.dspark_read_device_error.restype = I
        lib.dspark_status_string.argtypes = [I]
        lib.dspark_status_string.restype = ctypes.c_char_p
        lib.dspark_version.argtypes = []
        lib.dspark_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def check(fn: str, status: int) -> None:
    if status != 0:
        raise DsparkError(fn, status)
