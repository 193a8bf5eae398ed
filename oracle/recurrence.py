"""fp64 token-by-token oracle (ctypes wrapper of ``gdn_oracle.c``).  TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
module.  It follows the four steps of ``delta_rule`` in "Transformer by Hand,
ch. 7 -- Gated DeltaNet: the token-by-token recurrence" (section "The formula"
and the listing "qwen/deltanet.py"), in fp64, on inputs widened exactly from
their storage dtype.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

MODE_DELTA = 0
MODE_PLAIN_ADD = 1


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (fp64, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def bind(path: str):
    """Load a compiled oracle library and declare its entry points."""
    lib = ctypes.CDLL(path)
    d = ctypes.POINTER(ctypes.c_double)
    lib.gdn_oracle_forward.argtypes = [d, d, d, d, d, d, d, d, ctypes.POINTER(ctypes.c_int64),
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int]
    lib.gdn_oracle_forward.restype = ctypes.c_int
    lib.gdn_oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def use_library(lib) -> None:
    """Route this module's calls to another compiled copy (tests plant mistakes this way)."""
    global _lib
    with _lock:
        _lib = lib


def reset_library() -> None:
    global _lib
    with _lock:
        _lib = None


def max_threads() -> int:
    return int(_load().gdn_oracle_max_threads())


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def forward(q, k, v, g, beta, S0=None, cu_seqlens=None, scale: float = 1.0, mode: int = MODE_DELTA,
            normalize_qk: bool = False, threads: int = 0):
    """Run the recurrence.

    q, k: [B, T, Hqk, dk]; v: [B, T, Hv, dv]; g, beta: [B, T, Hv] (any float dtype,
    widened exactly to fp64).  With ``cu_seqlens`` (num_seqs+1 offsets) B must be 1
    and the T tokens are split into packed sequences.  S0: [num_seqs, Hv, dk, dv]
    or None (zeros).  Returns (out [B, T, Hv, dv] fp64, S_final [num_seqs, Hv, dk, dv] fp64).
    """
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    if cu_seqlens is None:
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        if B != 1:
            raise ValueError("packed sequences need B == 1")
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("cu_seqlens must rise from 0 to T")
    nseq = len(cu) - 1
    s0 = None if S0 is None else _f64(S0).reshape(nseq, Hv, dk, dv)
    out = np.zeros((B, T, Hv, dv), dtype=np.float64)
    sf = np.zeros((nseq, Hv, dk, dv), dtype=np.float64)
    rc = _load().gdn_oracle_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s0), _ptr(out),
                                    _ptr(sf), cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), nseq,
                                    Hqk, Hv, dk, dv, float(scale), int(mode), int(bool(normalize_qk)),
                                    int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle rejected its arguments (rc={rc})")
    return out, sf


def decode_step(q, k, v, g, beta, S, scale: float = 1.0, normalize_qk: bool = False,
                threads: int = 0):
    """One token per sequence: q, k [N, Hqk, dk]; v [N, Hv, dv]; g, beta [N, Hv];
    S [N, Hv, dk, dv].  Returns (out [N, Hv, dv], S_new [N, Hv, dk, dv]) in fp64."""
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    N = q.shape[0]
    out, sf = forward(q.reshape(1, N, *q.shape[1:]), k.reshape(1, N, *k.shape[1:]),
                      v.reshape(1, N, *v.shape[1:]), g.reshape(1, N, -1), beta.reshape(1, N, -1),
                      S0=S, cu_seqlens=np.arange(N + 1), scale=scale, normalize_qk=normalize_qk,
                      threads=threads)
    return out[0], sf
