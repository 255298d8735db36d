"""fp64 CPU oracle for the mLSTM cell (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path never does.

Every function takes array-likes (numpy arrays or CPU/GPU torch tensors),
widens them to contiguous float64 and calls the C routines in
``mlstm_oracle.c``; results come back as float64 numpy arrays.
See ``mlstm_oracle.c`` for the equations each routine evaluates.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build

_LIBS = {}
_D = ctypes.POINTER(ctypes.c_double)
_L = ctypes.POINTER(ctypes.c_long)


def _lib(mutation: int = 0) -> ctypes.CDLL:
    if mutation not in _LIBS:
        path = _build.build(mutation)
        lib = ctypes.CDLL(path)
        i, p = ctypes.c_int, _D
        lib.oracle_parallel_stabilized.argtypes = [i, i, i, i, i, p, p, p, p, p, p, p, p, p, i]
        lib.oracle_parallel_rows.argtypes = [i, i, i, i, i, p, p, p, p, p, p, _L, i, p, p, p, i]
        lib.oracle_parallel_unstabilized.argtypes = [i, i, i, i, i, p, p, p, p, p, p, p, i]
        lib.oracle_step.argtypes = [i, i, i, i, p, p, p, p, p, p, p, p, p, p, i]
        lib.oracle_recurrent_stabilized.argtypes = [i, i, i, i, i, p, p, p, p, p, p, p, p, p, p, i]
        lib.oracle_recurrent_unstabilized.argtypes = [i, i, i, i, i, p, p, p, p, p, p, p, i]
        lib.oracle_parallel_backward.argtypes = [i, i, i, i, i, p, p, p, p, p, p, p, p, p, p, p, i]
        lib.oracle_recurrent_backward.argtypes = [i, i, i, i, i] + [p] * 13 + [i]
        lib.oracle_recurrent_backward.restype = ctypes.c_int
        lib.oracle_set_forget_exp.argtypes = [i]
        lib.oracle_set_forget_exp.restype = None
        for f in ("oracle_parallel_stabilized", "oracle_parallel_rows", "oracle_parallel_backward",
                  "oracle_parallel_unstabilized", "oracle_step",
                  "oracle_recurrent_stabilized", "oracle_recurrent_unstabilized",
                  "oracle_mutation", "oracle_max_threads"):
            getattr(lib, f).restype = ctypes.c_int
        _LIBS[mutation] = lib
    return _LIBS[mutation]


def f64(x) -> np.ndarray:
    """Exact widening of an fp32/bf16/fp64 array-like to contiguous float64."""
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(_D)


def max_threads() -> int:
    return _lib().oracle_max_threads()


def _check(rc: int, name: str):
    if rc != 0:
        raise ValueError(f"{name}: invalid arguments (rc={rc})")


def parallel_stabilized(q, k, v, ig, fg, og=None, *, nthreads: int = 0, mutation: int = 0):
    """Stabilized parallel forward, eqs (79)-(86) [+ (78) if og].  Returns (h, m, n)."""
    q, k, v, ig, fg, og = map(f64, (q, k, v, ig, fg, og))
    B, H, T, dqk = q.shape
    dv = v.shape[-1]
    h = np.empty((B, H, T, dv))
    m = np.empty((B, H, T))
    n = np.empty((B, H, T))
    _check(_lib(mutation).oracle_parallel_stabilized(B, H, T, dqk, dv, _p(q), _p(k), _p(v), _p(ig), _p(fg),
                                                     _p(og), _p(h), _p(m), _p(n), nthreads), "parallel")
    return h, m, n


def parallel_rows(q, k, v, ig, fg, rows, og=None, *, nthreads: int = 0, mutation: int = 0):
    """Stabilized parallel forward for sampled rows; rows = flat indices bh*T + i.
    Returns (h [nrows,dv], m [nrows], n [nrows])."""
    q, k, v, ig, fg, og = map(f64, (q, k, v, ig, fg, og))
    B, H, T, dqk = q.shape
    dv = v.shape[-1]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nr = rows.shape[0]
    h = np.empty((nr, dv))
    m = np.empty(nr)
    n = np.empty(nr)
    _check(_lib(mutation).oracle_parallel_rows(B, H, T, dqk, dv, _p(q), _p(k), _p(v), _p(ig), _p(fg), _p(og),
                                               rows.ctypes.data_as(_L), nr, _p(h), _p(m), _p(n), nthreads),
           "parallel_rows")
    return h, m, n


def parallel_unstabilized(q, k, v, ig, fg, og=None, *, nthreads: int = 0, mutation: int = 0):
    """Unstabilized parallel forward, eqs (71)-(73), (76) [+ (78)]."""
    q, k, v, ig, fg, og = map(f64, (q, k, v, ig, fg, og))
    B, H, T, dqk = q.shape
    dv = v.shape[-1]
    h = np.empty((B, H, T, dv))
    _check(_lib(mutation).oracle_parallel_unstabilized(B, H, T, dqk, dv, _p(q), _p(k), _p(v), _p(ig), _p(fg),
                                                       _p(og), _p(h), nthreads), "parallel_unstabilized")
    return h


def recurrent_stabilized(q, k, v, ig, fg, og=None, *, nthreads: int = 0, mutation: int = 0):
    """Stabilized recurrence from C=0, n=0, m=-inf.  Returns (h, C_T, n_T, m_T)."""
    q, k, v, ig, fg, og = map(f64, (q, k, v, ig, fg, og))
    B, H, T, dqk = q.shape
    dv = v.shape[-1]
    h = np.empty((B, H, T, dv))
    C = np.empty((B, H, dv, dqk))
    n = np.empty((B, H, dqk))
    m = np.empty((B, H))
    _check(_lib(mutation).oracle_recurrent_stabilized(B, H, T, dqk, dv, _p(q), _p(k), _p(v), _p(ig), _p(fg),
                                                      _p(og), _p(h), _p(C), _p(n), _p(m), nthreads),
           "recurrent")
    return h, C, n, m


def recurrent_unstabilized(q, k, v, ig, fg, og=None, *, nthreads: int = 0, mutation: int = 0):
    q, k, v, ig, fg, og = map(f64, (q, k, v, ig, fg, og))
    B, H, T, dqk = q.shape
    dv = v.shape[-1]
    h = np.empty((B, H, T, dv))
    _check(_lib(mutation).oracle_recurrent_unstabilized(B, H, T, dqk, dv, _p(q), _p(k), _p(v), _p(ig),
                                                        _p(fg), _p(og), _p(h), nthreads),
           "recurrent_unstabilized")
    return h


class forget_exp:
    """Within the block, every oracle routine (of the given mutation build)
    uses the exponential forget activation log f = f~ instead of
    log sigma(f~) ("xLSTM", part 28/30: gamma is sigma or exp)."""

    def __init__(self, mutation: int = 0):
        self.lib = _lib(mutation)

    def __enter__(self):
        self.lib.oracle_set_forget_exp(1)
        return self

    def __exit__(self, *exc):
        self.lib.oracle_set_forget_exp(0)
        return False


def parallel_backward(q, k, v, ig, fg, dh, *, nthreads: int = 0, mutation: int = 0):
    """Gradients of the stabilized parallel forward (no output gate) for the
    output gradient dh = dL/dH~ [B,H,T,d_v]: returns (dq, dk, dv, d_igate,
    d_fgate) in fp64, following part 28/30 eqs (87)-(105)."""
    q, k, v, ig, fg, dh = map(f64, (q, k, v, ig, fg, dh))
    B, H, T, dqk = q.shape
    dv = v.shape[-1]
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dvv = np.empty_like(v)
    dig = np.empty((B, H, T))
    dfg = np.empty((B, H, T))
    _check(_lib(mutation).oracle_parallel_backward(B, H, T, dqk, dv, _p(q), _p(k), _p(v), _p(ig), _p(fg), _p(dh),
                                                   _p(dq), _p(dk), _p(dvv), _p(dig), _p(dfg), nthreads),
           "parallel_backward")
    return dq, dk, dvv, dig, dfg


def recurrent_backward(q, k, v, ig, fg, dh, og=None, *, nthreads: int = 0, mutation: int = 0):
    """Backpropagation through time of the unstabilized recurrence (part 28/30
    eqs 59-70) for dh = dL/dh [B,H,T,d_v]: returns (dq, dk, dv, d_igate,
    d_fgate, d_ogate) in fp64 (d_ogate None without an output gate)."""
    q, k, v, ig, fg, dh, og = map(f64, (q, k, v, ig, fg, dh, og))
    B, H, T, dqk = q.shape
    dv = v.shape[-1]
    dq, dk, dvv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    dig, dfg = np.empty((B, H, T)), np.empty((B, H, T))
    dog = np.empty_like(dh) if og is not None else None
    _check(_lib(mutation).oracle_recurrent_backward(B, H, T, dqk, dv, _p(q), _p(k), _p(v), _p(ig), _p(fg), _p(og),
                                                    _p(dh), _p(dq), _p(dk), _p(dvv), _p(dig), _p(dfg), _p(dog),
                                                    nthreads), "recurrent_backward")
    return dq, dk, dvv, dig, dfg, dog


def step_seq(C, n, m, q, k, v, ig, fg, o=None, *, nthreads: int = 0, mutation: int = 0):
    """L consecutive stabilized steps on copies of the given state: ``step``
    applied to tokens t = 0..L-1 in order (q, k [B,H,L,d_qk], v, o [B,H,L,d_v],
    ig, fg [B,H,L]).  Returns (h [B,H,L,d_v], C, n, m) after the last token."""
    C, n, m = f64(C).copy(), f64(n).copy(), f64(m).copy()
    q, k, v, ig, fg, o = map(f64, (q, k, v, ig, fg, o))
    B, H, L, _ = q.shape
    h = np.empty((B, H, L, v.shape[-1]))
    for t in range(L):
        h[:, :, t], C, n, m = step(C, n, m, q[:, :, t], k[:, :, t], v[:, :, t], ig[:, :, t], fg[:, :, t],
                                   None if o is None else o[:, :, t], nthreads=nthreads, mutation=mutation)
    return h, C, n, m


def step(C, n, m, q, k, v, ig, fg, o=None, *, nthreads: int = 0, mutation: int = 0):
    """One stabilized recurrent step on copies of the given state.
    Returns (h, C_new, n_new, m_new); the inputs are not modified."""
    C, n, m, q, k, v, ig, fg, o = map(f64, (C, n, m, q, k, v, ig, fg, o))
    C, n, m = C.copy(), n.copy(), m.copy()
    B, H, dqk = q.shape
    dv = v.shape[-1]
    h = np.empty((B, H, dv))
    _check(_lib(mutation).oracle_step(B, H, dqk, dv, _p(C), _p(n), _p(m), _p(q), _p(k), _p(v), _p(o),
                                      _p(ig), _p(fg), _p(h), nthreads), "step")
    return h, C, n, m
