"""Build and load the oracle's C model (``exp2_model.c``) -- TEST INFRASTRUCTURE ONLY.

``build()`` compiles it with gcc into ``oracle/liboracle_exp2.so``; it is called
by ``__graft_entry__.build()`` and, lazily, by ``exp2_emulated`` when the shared
object is missing or older than the source. The model is plain C with no
architecture-specific flags, so it gives the same bits on x86-64 and aarch64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "exp2_model.c")
_LIB = os.path.join(_HERE, "liboracle_exp2.so")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-frounding-math",
               "-ffp-contract=off", "-fno-fast-math", "-o", _LIB, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_exp2_emulated.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_long]
        lib.oracle_exp2_emulated.restype = None
        _lib = lib
    return _lib


def exp2_emulated(x) -> np.ndarray:
    """Software exp2 of float32 inputs through the scalar C model."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    y = np.empty_like(x)
    _load().oracle_exp2_emulated(x.ctypes.data, y.ctypes.data, x.size)
    return y
