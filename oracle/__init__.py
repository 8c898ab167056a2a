"""fp64 CPU oracle for bounded-decay gated linear attention — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The CUDA library never does, and this
package imports nothing from it.

The arithmetic lives in ``bdla_oracle.c`` (token-by-token recurrence and its
reverse mode, see the header there for the reading of the pages; the
per-channel decay variant is ``fwd_vec`` / ``bwd_vec``, the gated delta
rule ``fwd_delta`` / ``bwd_delta``).  This module
only compiles it with gcc and marshals numpy float64 arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bdla_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BOUNDED = 0    # lambda = b * sigmoid(a)
SOFTPLUS = 1   # lambda = -softplus(a)  (unbounded ablation)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP) into oracle/liboracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            lib.oracle_fwd.argtypes = [ctypes.c_int, i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       dp, dp, dp, dp, ctypes.c_double, ctypes.c_int, dp, dp, dp,
                                       ctypes.c_int]
            lib.oracle_fwd.restype = ctypes.c_int
            lib.oracle_bwd.argtypes = [ctypes.c_int, i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       dp, dp, dp, dp, ctypes.c_double, ctypes.c_int, dp,
                                       dp, dp, dp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_int]
            lib.oracle_bwd.restype = ctypes.c_int
            lib.oracle_fwd_vec.argtypes = lib.oracle_fwd.argtypes
            lib.oracle_fwd_vec.restype = ctypes.c_int
            lib.oracle_bwd_vec.argtypes = lib.oracle_bwd.argtypes
            lib.oracle_bwd_vec.restype = ctypes.c_int
            lib.oracle_fwd_delta.argtypes = [ctypes.c_int, i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             dp, dp, dp, dp, dp, ctypes.c_double, ctypes.c_int, dp, dp, dp,
                                             ctypes.c_int]
            lib.oracle_fwd_delta.restype = ctypes.c_int
            lib.oracle_bwd_delta.argtypes = [ctypes.c_int, i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             dp, dp, dp, dp, dp, ctypes.c_double, ctypes.c_int, dp,
                                             dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_int]
            lib.oracle_bwd_delta.restype = ctypes.c_int
            lib.oracle_log_decay.argtypes = [ctypes.c_int64, dp, ctypes.c_double, ctypes.c_int, dp]
            lib.oracle_log_decay.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    x = np.ascontiguousarray(x, dtype=np.float64)
    return x


def _ptr(x):
    if x is None:
        return None
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _cu(cu_seqlens, T):
    if cu_seqlens is None:
        cu_seqlens = [0, T]
    return np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))


def log_decay(a, b=-5.0, mode=BOUNDED):
    a = _f64(a)
    out = np.empty_like(a)
    _load().oracle_log_decay(a.size, _ptr(a), float(b), int(mode), _ptr(out))
    return out


def fwd(q, k, v, a, b=-5.0, mode=BOUNDED, h0=None, cu_seqlens=None, nthreads=0):
    """Forward recurrence.  q,k [T,H,dk], v [T,H,dv], a [T,H] (packed
    documents given by cu_seqlens, default one document).  Returns (o, hT)
    with o [T,H,dv] and hT [N,H,dk,dv], all float64."""
    q, k, v, a, h0 = _f64(q), _f64(k), _f64(v), _f64(a), _f64(h0)
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = cu.size - 1
    assert cu[0] == 0 and cu[-1] == T
    o = np.zeros((T, H, dv))
    hT = np.zeros((N, H, dk, dv))
    _load().oracle_fwd(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, dk, dv,
                       _ptr(q), _ptr(k), _ptr(v), _ptr(a), float(b), int(mode), _ptr(h0),
                       _ptr(o), _ptr(hT), int(nthreads))
    return o, hT


def bwd(q, k, v, a, dO, b=-5.0, mode=BOUNDED, h0=None, dhT=None, cu_seqlens=None,
        window=1024, nthreads=0):
    """Reverse mode of ``fwd`` for the loss <o, dO> + <hT, dhT>.  Returns
    (dq, dk, dv, da, dh0), float64."""
    q, k, v, a, dO, h0, dhT = (_f64(x) for x in (q, k, v, a, dO, h0, dhT))
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = cu.size - 1
    dq = np.zeros_like(q)
    dkk = np.zeros_like(k)
    dvv = np.zeros_like(v)
    da = np.zeros_like(a)
    dh0 = np.zeros((N, H, dk, dv))
    _load().oracle_bwd(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, dk, dv,
                       _ptr(q), _ptr(k), _ptr(v), _ptr(a), float(b), int(mode), _ptr(h0),
                       _ptr(dO), _ptr(dhT), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(da),
                       _ptr(dh0), int(window), int(nthreads))
    return dq, dkk, dvv, da, dh0


def fwd_vec(q, k, v, a, b=-5.0, mode=BOUNDED, h0=None, cu_seqlens=None, nthreads=0):
    """Forward recurrence with one log-decay per key channel:
    S_t = diag(exp(lambda_t)) S_{t-1} + k_t v_t^T.  a [T,H,dk]; otherwise as
    ``fwd``.  Returns (o, hT), float64."""
    q, k, v, a, h0 = _f64(q), _f64(k), _f64(v), _f64(a), _f64(h0)
    T, H, dk = q.shape
    dv = v.shape[2]
    assert a.shape == (T, H, dk)
    cu = _cu(cu_seqlens, T)
    N = cu.size - 1
    assert cu[0] == 0 and cu[-1] == T
    o = np.zeros((T, H, dv))
    hT = np.zeros((N, H, dk, dv))
    _load().oracle_fwd_vec(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, dk, dv,
                           _ptr(q), _ptr(k), _ptr(v), _ptr(a), float(b), int(mode), _ptr(h0),
                           _ptr(o), _ptr(hT), int(nthreads))
    return o, hT


def bwd_vec(q, k, v, a, dO, b=-5.0, mode=BOUNDED, h0=None, dhT=None, cu_seqlens=None,
            window=1024, nthreads=0):
    """Reverse mode of ``fwd_vec`` for the loss <o, dO> + <hT, dhT>.  Returns
    (dq, dk, dv, da, dh0) with da [T,H,dk], float64."""
    q, k, v, a, dO, h0, dhT = (_f64(x) for x in (q, k, v, a, dO, h0, dhT))
    T, H, dk = q.shape
    dv = v.shape[2]
    assert a.shape == (T, H, dk)
    cu = _cu(cu_seqlens, T)
    N = cu.size - 1
    dq = np.zeros_like(q)
    dkk = np.zeros_like(k)
    dvv = np.zeros_like(v)
    da = np.zeros_like(a)
    dh0 = np.zeros((N, H, dk, dv))
    _load().oracle_bwd_vec(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, dk, dv,
                           _ptr(q), _ptr(k), _ptr(v), _ptr(a), float(b), int(mode), _ptr(h0),
                           _ptr(dO), _ptr(dhT), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(da),
                           _ptr(dh0), int(window), int(nthreads))
    return dq, dkk, dvv, da, dh0


def fwd_delta(q, k, v, a, beta, b=-5.0, mode=BOUNDED, h0=None, cu_seqlens=None, nthreads=0):
    """Gated delta rule with the bounded log-decay:
    S_t = g_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T, o_t = S_t^T q_t.
    beta [T,H] (write strengths, given); otherwise as ``fwd``.  Returns
    (o, hT), float64."""
    q, k, v, a, beta, h0 = _f64(q), _f64(k), _f64(v), _f64(a), _f64(beta), _f64(h0)
    T, H, dk = q.shape
    dv = v.shape[2]
    assert a.shape == (T, H) and beta.shape == (T, H)
    cu = _cu(cu_seqlens, T)
    N = cu.size - 1
    assert cu[0] == 0 and cu[-1] == T
    o = np.zeros((T, H, dv))
    hT = np.zeros((N, H, dk, dv))
    _load().oracle_fwd_delta(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, dk, dv,
                             _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), float(b), int(mode),
                             _ptr(h0), _ptr(o), _ptr(hT), int(nthreads))
    return o, hT


def bwd_delta(q, k, v, a, beta, dO, b=-5.0, mode=BOUNDED, h0=None, dhT=None, cu_seqlens=None,
              window=1024, nthreads=0):
    """Reverse mode of ``fwd_delta`` for the loss <o, dO> + <hT, dhT>.
    Returns (dq, dk, dv, da, dbeta, dh0), float64."""
    q, k, v, a, beta, dO, h0, dhT = (_f64(x) for x in (q, k, v, a, beta, dO, h0, dhT))
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = cu.size - 1
    dq = np.zeros_like(q)
    dkk = np.zeros_like(k)
    dvv = np.zeros_like(v)
    da = np.zeros_like(a)
    dbeta = np.zeros_like(beta)
    dh0 = np.zeros((N, H, dk, dv))
    _load().oracle_bwd_delta(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, dk, dv,
                             _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), float(b), int(mode),
                             _ptr(h0), _ptr(dO), _ptr(dhT), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(da),
                             _ptr(dbeta), _ptr(dh0), int(window), int(nthreads))
    return dq, dkk, dvv, da, dbeta, dh0


def threads_used(nthreads=0):
    """Thread count the oracle would use (OpenMP max threads)."""
    lib = _load()
    q = np.zeros((1, 1, 1))
    a = np.zeros((1, 1))
    o = np.zeros((1, 1, 1))
    hT = np.zeros((1, 1, 1, 1))
    cu = np.array([0, 1], dtype=np.int64)
    return lib.oracle_fwd(1, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), 1, 1, 1,
                          _ptr(q), _ptr(q), _ptr(q), _ptr(a), -5.0, 0, None, _ptr(o), _ptr(hT),
                          int(nthreads))
