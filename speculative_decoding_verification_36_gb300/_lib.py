"""ctypes loader for libspecverify.so (the C ABI of include/specverify.h).

The library is built in-tree by ``build.py`` (``__graft_entry__.build()``).
Loading fails loudly when it is missing: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libspecverify.so")
HEADER = os.path.join(ROOT, "include", "specverify.h")

SPEC_OK = 0
SPEC_ERR_NULL = -1
SPEC_ERR_SHAPE = -2
SPEC_ERR_TEMPERATURE = -3
SPEC_ERR_CUDA = -4
SPEC_ERR_SCRATCH = -5
SPEC_ERR_HINT = -6
SPEC_STATIC_SCRATCH_BYTES = 8 << 20
SPEC_FLAG_BAD_DATA = 1
SPEC_FLAG_TIMEOUT = 2

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_U64 = ctypes.c_uint64
_D = ctypes.c_double

# name -> argtypes (restype is int for all but spec_status_string)
SIGNATURES = {
    "spec_verify_f32": [_P, _P, _P, _I, _I, _I, _F, _U64, _P, _P, _P],
    "spec_verify_bf16": [_P, _P, _P, _I, _I, _I, _F, _U64, _P, _P, _P],
    "spec_verify_bf16_static_scratch": [_P, _P, _P, _I, _I, _I, _F, _U64, _P, _P, _P],
    "spec_verify_early_exit_f32": [_P, _P, _P, _I, _I, _I, _F, _U64, _P, _P, _P],
    "spec_verify_early_exit_bf16": [_P, _P, _P, _I, _I, _I, _F, _U64, _P, _P, _P],
    "spec_verify_stats_f32": [_P, _P, _P, _I, _I, _I, _F, _U64, _P, _P, _P, _P, _P, _P, _P],
    "spec_verify_stats_bf16": [_P, _P, _P, _I, _I, _I, _F, _U64, _P, _P, _P, _P, _P, _P, _P],
    "spec_verify_khint_f32": [_P, _P, _P, _I, _I, _I, _F, _U64, _D, _D, _I, _I, _P, _P, _P, _P, _P],
    "spec_verify_khint_bf16": [_P, _P, _P, _I, _I, _I, _F, _U64, _D, _D, _I, _I, _P, _P, _P, _P, _P],
    "spec_verify_greedy_argmax_f32": [_P, _P, _I, _I, _I, _P, _P, _P, _P],
    "spec_verify_greedy_argmax_bf16": [_P, _P, _I, _I, _I, _P, _P, _P, _P],
    "spec_tree_verify_greedy_f32": [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P],
    "spec_tree_verify_greedy_bf16": [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P],
    "spec_tree_verify_greedy_early_exit_f32": [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P],
    "spec_tree_verify_greedy_early_exit_bf16": [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P],
    "spec_tree_verify_sampling_f32": [_P, _P, _P, _P, _I, _I, _I, _F, _U64, _P, _P, _P],
    "spec_tree_verify_sampling_bf16": [_P, _P, _P, _P, _I, _I, _I, _F, _U64, _P, _P, _P],
    "spec_acceptance_stats": [_P, _I, _I, _P, _P, _P, _P],
    "spec_ngram_draft": [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P],
    "spec_test_fail_allocations": [_I],
    "spec_test_spin_limit": [ctypes.c_uint32],
    "spec_test_wait_probe": [ctypes.c_void_p],
    "spec_get_status": [_P, _P],
    "spec_status_string": [_I],
}


class SpecError(RuntimeError):
    """A non-zero return code from libspecverify."""

    def __init__(self, code: int, message: str):
        super().__init__(f"libspecverify error {code}: {message}")
        self.code = code


def header_symbols(path: str = HEADER):
    """Function names declared in include/specverify.h."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:int|const char\s*\*)\s*\*?\s*(spec_\w+)\s*\(", text, flags=re.M)


def load():
    """Load libspecverify.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                f"g.build()'` (needs nvcc).  There is no CPU fallback.")
        lib = ctypes.CDLL(LIB_PATH)
        for name, argtypes in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = argtypes
            fn.restype = ctypes.c_char_p if name == "spec_status_string" else ctypes.c_int
        _lib = lib
        return lib


def check(code: int) -> None:
    if code != SPEC_OK:
        msg = load().spec_status_string(code)
        raise SpecError(code, msg.decode() if msg else "?")
