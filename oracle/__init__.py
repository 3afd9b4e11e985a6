"""float64 CPU oracle for the GDN forward.  TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's cpu_baseline leg may
import this package.  It shares no code with the CUDA path and never imports
it.

* ``recurrence``       -- the token-by-token gated delta rule (plain C, pthreads).
* ``chunked``          -- the chunked closed form and the context-parallel
                          combine (numpy), used to pin the recurrence and to
                          give warmup-mode expectations.
* ``backward``         -- gradients of the forward: autograd of the token
                          recurrence (the definition) and the chunk-level
                          derivation the GPU backward follows (numpy).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the C oracle with gcc (plain -O2, no fast-math, no contraction)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    f = lib.gdn_oracle_recurrence
    dp = ctypes.POINTER(ctypes.c_double)
    f.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int64), ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_double, dp, dp, dp, dp, dp, dp, dp, dp,
                  ctypes.POINTER(ctypes.c_int32), ctypes.c_int]
    f.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(path)
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = _bind(_LIB_PATH)
    return _lib


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a, ctype=ctypes.c_double):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def recurrence(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None, heads=None,
               n_threads=None, want_state=True, lib=None):
    """Token-by-token float64 gated delta rule.

    q,k [T, h_qk, d_k]; v [T, h_v, d_v]; g,beta [T, h_v]; h0 [N, h_v, d_k, d_v] or None.
    cu_seqlens: N+1 token offsets (None: one sequence of T tokens).
    heads: iterable of value heads to compute (None: all); other heads' outputs stay 0.
    Returns (o [T, h_v, d_v], hT [N, h_v, d_k, d_v] or None), float64.
    """
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    T, h_qk, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    if cu_seqlens is None:
        cu_seqlens = [0, T]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    n_seqs = len(cu) - 1
    if scale is None:
        scale = 1.0 / np.sqrt(d_k)
    mask = None
    if heads is not None:
        mask = np.zeros(h_v, dtype=np.int32)
        mask[list(heads)] = 1
    o = np.zeros((T, h_v, d_v))
    hT = np.zeros((n_seqs, h_v, d_k, d_v)) if want_state else None
    lib = lib or load()
    rc = lib.gdn_oracle_recurrence(
        n_seqs, _ptr(cu, ctypes.c_int64), h_qk, h_v, d_k, d_v, float(scale),
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(hT),
        _ptr(mask, ctypes.c_int32), int(n_threads or default_threads()))
    if rc != 0:
        raise ValueError("gdn_oracle_recurrence rejected its arguments")
    return o, hT
