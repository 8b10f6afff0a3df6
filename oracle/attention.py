"""Oracle attention (test infrastructure only): loader and wrappers for attention_ref.c.

``build()`` compiles the plain C oracle with gcc into ``oracle/_build/liboracle.so``;
``attention_rows`` calls it.  Nothing here touches a GPU or the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_ref.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc -O2 -fopenmp).  Returns the library path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC,
                               "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_attention_rows.argtypes = [
            ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
        lib.oracle_max_threads.restype = ctypes.c_int32
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def attention_rows(q, pos, k, v, scale, num_threads: int = 0):
    """Causal attention of query rows over one request's logical-order keys/values.

    q: [n, hq, d] float32; pos: [n] absolute positions (row attends keys 0..pos);
    k, v: [L, hkv, d] float32.  Returns (out [n, hq, d] float32, lse [n, hq] float64).
    """
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    n, hq, d = q.shape
    L, hkv, d2 = k.shape
    assert d2 == d and v.shape == k.shape and pos.shape == (n,)
    out = np.empty((n, hq, d), np.float32)
    lse = np.empty((n, hq), np.float64)
    rc = _load().oracle_attention_rows(n, hq, hkv, d, L, q.ctypes.data, pos.ctypes.data,
                                       k.ctypes.data, v.ctypes.data, float(scale),
                                       out.ctypes.data, lse.ctypes.data, int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle_attention_rows failed with {rc}")
    return out, lse
