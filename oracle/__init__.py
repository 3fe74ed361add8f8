"""fp64 CPU oracle for exact softmax attention (forward and backward).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library never
imports, links or runs anything here, and this package imports nothing from
the CUDA side.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over independent
(sequence, head) units); this module only compiles it and marshals numpy
arrays through ctypes.  Every function takes and returns float64 arrays in the
layouts documented in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, -O2, OpenMP, IEEE math)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            common = [ctypes.c_int] * 6 + [ctypes.c_double] + [ctypes.c_int] * 3 + [dp, ip, ip]
            lib.oracle_fwd.argtypes = common + [dp] * 6
            lib.oracle_fwd.restype = ctypes.c_int
            lib.oracle_bwd.argtypes = common + [dp] * 8
            lib.oracle_bwd.restype = ctypes.c_int
            lib.oracle_threads.argtypes = []
            lib.oracle_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle runs with."""
    return int(_load().oracle_threads())


def _dptr(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(a):
    if a is None:
        return None
    assert a.dtype == np.int32 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _prep(q, k, v, sinks, cu_q, cu_k):
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    sinks = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float64)
    cu_q = None if cu_q is None else np.ascontiguousarray(cu_q, dtype=np.int32)
    cu_k = None if cu_k is None else np.ascontiguousarray(cu_k, dtype=np.int32)
    return q, k, v, sinks, cu_q, cu_k


def _dims(q, k, cu_q, cu_k):
    """(B, s_q, s_kv, h_q, h_kv, d) from array shapes (dense 4-D or packed 3-D)."""
    if cu_q is None:
        B, s_q, h_q, d = q.shape
        _, s_kv, h_kv, _ = k.shape
    else:
        _, h_q, d = q.shape
        _, h_kv, _ = k.shape
        B = len(cu_q) - 1
        s_q, s_kv = int(cu_q[-1]), int(cu_k[-1])
    return B, s_q, s_kv, h_q, h_kv, d


def fwd(q, k, v, *, scale=None, causal=False, window=(-1, -1), sinks=None, cu_q=None, cu_k=None):
    """Forward: returns (o, lse, lse_nosink) in fp64.

    q: [B, s_q, h_q, d] or packed [T_q, h_q, d]; k, v: [B, s_kv, h_kv, d] or
    [T_k, h_kv, d]; sinks: [h_q] or None; cu_q, cu_k: int32 [B+1] or None.
    lse / lse_nosink: [B, h_q, s_q] dense, [h_q, T_q] packed.
    """
    q, k, v, sinks, cu_q, cu_k = _prep(q, k, v, sinks, cu_q, cu_k)
    B, s_q, s_kv, h_q, h_kv, d = _dims(q, k, cu_q, cu_k)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.zeros_like(q)
    lshape = (B, h_q, s_q) if cu_q is None else (h_q, s_q)
    lse = np.zeros(lshape, np.float64)
    lse0 = np.zeros(lshape, np.float64)
    rc = _load().oracle_fwd(B, s_q, s_kv, h_q, h_kv, d, float(scale), int(bool(causal)),
                            int(window[0]), int(window[1]), _dptr(sinks), _iptr(cu_q), _iptr(cu_k),
                            _dptr(q), _dptr(k), _dptr(v), _dptr(o), _dptr(lse), _dptr(lse0))
    if rc != 0:
        raise ValueError(f"oracle_fwd rejected its arguments (code {rc})")
    return o, lse, lse0


def bwd(q, k, v, dout, *, scale=None, causal=False, window=(-1, -1), sinks=None, cu_q=None,
        cu_k=None):
    """Backward of sum(O * dout): returns (dq, dk, dv, dsinks) in fp64 (dsinks None without sinks)."""
    q, k, v, sinks, cu_q, cu_k = _prep(q, k, v, sinks, cu_q, cu_k)
    dout = np.ascontiguousarray(dout, dtype=np.float64)
    B, s_q, s_kv, h_q, h_kv, d = _dims(q, k, cu_q, cu_k)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dsinks = None if sinks is None else np.zeros(h_q, np.float64)
    rc = _load().oracle_bwd(B, s_q, s_kv, h_q, h_kv, d, float(scale), int(bool(causal)),
                            int(window[0]), int(window[1]), _dptr(sinks), _iptr(cu_q), _iptr(cu_k),
                            _dptr(q), _dptr(k), _dptr(v), _dptr(dout), _dptr(dq), _dptr(dk),
                            _dptr(dv), _dptr(dsinks))
    if rc != 0:
        raise ValueError(f"oracle_bwd rejected its arguments (code {rc})")
    return dq, dk, dv, dsinks
