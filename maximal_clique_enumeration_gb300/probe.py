"""Binding of libmce_probe.so: the measured rate of the search's inner integer operation."""
from __future__ import annotations

import ctypes
import os

from .build import PROBE_PATH

_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(PROBE_PATH):
            raise RuntimeError(f"{PROBE_PATH} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(PROBE_PATH)
        lib.mce_probe_word_rate.restype = ctypes.c_int
        lib.mce_probe_word_rate.argtypes = [ctypes.c_int, ctypes.c_int,
                                            ctypes.POINTER(ctypes.c_double),
                                            ctypes.POINTER(ctypes.c_float)]
        _lib = lib
    return _lib


def word_rate(iters: int = 20000, reps: int = 5) -> dict:
    """Sustained AND + popcount + accumulate rate on 32-bit words (words per second)."""
    rate = ctypes.c_double(0.0)
    ms = ctypes.c_float(0.0)
    code = _load().mce_probe_word_rate(iters, reps, ctypes.byref(rate), ctypes.byref(ms))
    if code:
        raise RuntimeError(f"mce_probe_word_rate failed with status {code}")
    return {"words_per_s": rate.value, "ms": ms.value}
