"""fp64 CPU oracle for the KDA recurrence -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its binding) never does, and shares no code with it.

The arithmetic lives in ``kda_oracle.c`` (plain C, fp64, sequential loops per
(sequence, head); threads only over independent units). This module compiles
it with gcc and marshals numpy arrays into it. Every input is converted to
float64 exactly (bf16 and fp32 values upcast without rounding).

Citations (web page titles and sections) are in ``kda_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` (gcc, -O2, no fast-math, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-fopenmp", "-shared",
           "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            ci, cd = ctypes.c_int, ctypes.c_double
            lib.oracle_shortconv_step.argtypes = [dp, dp, dp, dp, ci, ci, ci]
            lib.oracle_shortconv_seq.argtypes = [dp, dp, dp, dp, dp, ctypes.c_void_p, ci,
                                                 ctypes.c_int64, ci, ci]
            lib.oracle_shortconv_step.restype = None
            lib.oracle_recurrence.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp,
                                              i64p, ci, ci, ci, cd, ci]
            lib.oracle_recurrence.restype = None
            lib.oracle_chunked.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp,
                                           i64p, ci, ci, ci, cd, ci, ci]
            lib.oracle_chunked.restype = None
            lib.oracle_gated_rmsnorm.argtypes = [dp, dp, dp, dp, ctypes.c_int64, ci, cd, ci]
            lib.oracle_gated_rmsnorm.restype = None
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ci
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def shortconv_step(x, ring, w):
    """One short-conv decode step. Returns (y, new_ring); inputs untouched.

    x [B,3,H,D], ring [B,3,H,3,D] (chronological, slot 0 oldest),
    w [3,H,D,4] (tap 3 multiplies the current token).
    """
    x = _f64(x)
    ring = _f64(ring).copy()
    w = _f64(w)
    B, P, H, D = x.shape
    assert P == 3 and ring.shape == (B, 3, H, 3, D) and w.shape == (3, H, D, 4)
    y = np.empty_like(x)
    _load().oracle_shortconv_step(_ptr(x), _ptr(ring), _ptr(w), _ptr(y), B, H, D)
    return y, ring


def shortconv_seq(x, w, ring_in=None, cu_seqlens=None):
    """Short conv over packed sequences. Returns (y [3,T,H,D], ring_out [N,3,H,3,D]).

    x [T,3,H,D]; w [3,H,D,4]; ring_in [N,3,H,3,D] or None (zero history);
    cu_seqlens [N+1] or None (one sequence of T tokens).
    """
    x = _f64(x)
    w = _f64(w)
    T, P, H, D = x.shape
    assert P == 3 and w.shape == (3, H, D, 4)
    cu = _seqlens(cu_seqlens, T)
    N = len(cu) - 1
    rin = None
    if ring_in is not None:
        rin = _f64(ring_in)
        assert rin.shape == (N, 3, H, 3, D)
    y = np.empty((3, T, H, D))
    rout = np.empty((N, 3, H, 3, D))
    _load().oracle_shortconv_seq(_ptr(x), _ptr(rin) if rin is not None else None, _ptr(w), _ptr(y),
                                 _ptr(rout), cu.ctypes.data_as(ctypes.c_void_p), N, T, H, D)
    return y, rout


def _seqlens(cu_seqlens, T):
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int64)
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    assert cu[0] == 0 and cu[-1] == T and np.all(np.diff(cu) >= 0)
    return cu


def recurrence(q, k, v, g, beta, s_init=None, cu_seqlens=None, eps=1e-6,
               nthreads=1, chunk=None):
    """Token-by-token KDA recurrence (or, with ``chunk=C``, its chunked form).

    q,k,v,g [T,H,D]; beta [T,H]; s_init [N,H,D,D] or None (zeros);
    cu_seqlens [N+1] or None (one sequence). Returns (out [T,H,D], s_final).
    """
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    T, H, D = q.shape
    assert k.shape == v.shape == g.shape == (T, H, D) and beta.shape == (T, H)
    cu = _seqlens(cu_seqlens, T)
    N = len(cu) - 1
    si = None
    if s_init is not None:
        si = _f64(s_init)
        assert si.shape == (N, H, D, D)
    out = np.zeros((T, H, D), dtype=np.float64)
    sf = np.zeros((N, H, D, D), dtype=np.float64)
    cup = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    lib = _load()
    if chunk is None:
        lib.oracle_recurrence(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                              _ptr(si), _ptr(sf), _ptr(out), cup, N, H, D,
                              float(eps), int(nthreads))
    else:
        lib.oracle_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           _ptr(si), _ptr(sf), _ptr(out), cup, N, H, D,
                           float(eps), int(chunk), int(nthreads))
    return out, sf


def decode_step(q, k, v, g, beta, state, eps=1e-6, nthreads=1):
    """One decode step for B sequences: q,k,v,g [B,H,D], beta [B,H],
    state [B,H,D,D]. Returns (out [B,H,D], new_state)."""
    B = np.asarray(q).shape[0]
    cu = np.arange(B + 1, dtype=np.int64)
    return recurrence(q, k, v, g, beta, s_init=state, cu_seqlens=cu, eps=eps,
                      nthreads=nthreads)


def gated_rmsnorm(o, gate, weight, eps=1e-6, act="sigmoid"):
    """Output epilogue: o, gate [..., D] (one row per token-head), weight [D].
    Returns y [..., D] = RMSNorm(o) * weight * act(gate), act in
    {"sigmoid", "silu"}."""
    o, gate, weight = _f64(o), _f64(gate), _f64(weight)
    assert o.shape == gate.shape and weight.shape == (o.shape[-1],)
    D = o.shape[-1]
    R = o.size // D if D else 0
    y = np.empty_like(o)
    _load().oracle_gated_rmsnorm(_ptr(o), _ptr(gate), _ptr(weight), _ptr(y), R, D, float(eps),
                                 {"sigmoid": 0, "silu": 1}[act])
    return y
