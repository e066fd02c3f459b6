"""ctypes wrapper of ``canon_f32.c`` (the canonical float32 index score).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  ``build()`` compiles
the C file with gcc; nothing here touches the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "canon_f32.c")
_LIB = os.path.join(_HERE, "liboracle_canon.so")
_handle = None


def build(force: bool = False) -> str:
    """Compile the oracle's C part (gcc, no fp contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared",
                               "-fPIC", "-o", _LIB, _SRC, "-lm"])
    return _LIB


def _lib():
    global _handle
    if _handle is None:
        _handle = ctypes.CDLL(build())
        f = _handle.oracle_index_scores_f32
        f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 3 + [ctypes.c_void_p]
        f.restype = None
    return _handle


def index_scores_f32(q_idx, w, k_idx) -> np.ndarray:
    """q_idx [H_I, d_I], w [H_I], k_idx [N, d_I] (all float32) -> float32 [N]."""
    q = np.ascontiguousarray(q_idx, dtype=np.float32)
    ww = np.ascontiguousarray(w, dtype=np.float32)
    k = np.ascontiguousarray(k_idx, dtype=np.float32).reshape(-1, q.shape[1])
    out = np.empty(k.shape[0], dtype=np.float32)
    _lib().oracle_index_scores_f32(q.ctypes.data, ww.ctypes.data, k.ctypes.data,
                                   q.shape[0], q.shape[1], k.shape[0], out.ctypes.data)
    return out
