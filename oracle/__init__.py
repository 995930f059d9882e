"""Plain fp64 CPU oracle for causal log-linear Mamba-2 attention and for the
log-linear Gated DeltaNet.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(the ``log_linear_attention_gb300`` package and its CUDA library) never does.

The arithmetic lives in ``lla_oracle.c`` (single-threaded, fp64, written as
the definition reads); this module only compiles it with gcc and marshals
numpy arrays through ctypes. Sources: "Log-Linear Attention" (gist.science
summaries of arXiv 2506.04761), §2 of the Portuguese and French pages
(Fenwick partition, hierarchical mask M_H, recurrent and chunkwise forms).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lla_oracle.c")
_LIB = os.path.join(_HERE, "liblla_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``lla_oracle.c`` into ``liblla_oracle.so`` next to it."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            lib.lla_oracle_level.argtypes = [ctypes.c_int64, ctypes.c_int64]
            lib.lla_oracle_level.restype = ctypes.c_int
            lib.lla_oracle_num_levels.argtypes = [ctypes.c_int64]
            lib.lla_oracle_num_levels.restype = ctypes.c_int
            lib.lla_oracle_explicit.argtypes = [dp] * 6 + [ctypes.c_int] * 6
            lib.lla_oracle_explicit.restype = None
            lib.lla_oracle_recurrent.argtypes = [dp] * 6 + [ctypes.c_int] * 6
            lib.lla_oracle_recurrent.restype = ctypes.c_int
            lib.lla_oracle_explicit_rows.argtypes = [dp] * 6 + [ctypes.c_int] * 5 + [i64p, ctypes.c_int]
            lib.lla_oracle_explicit_rows.restype = None
            lib.lla_oracle_decode_step.argtypes = [dp] * 6 + [i64p, dp] + [ctypes.c_int] * 5
            lib.lla_oracle_decode_step.restype = ctypes.c_int
            lib.lla_oracle_backward.argtypes = [dp] * 11 + [ctypes.c_int] * 6
            lib.lla_oracle_backward.restype = None
            lib.lla_oracle_backward_rows.argtypes = [dp] * 6 + [ctypes.c_int] * 5 + [i64p, ctypes.c_int] + [dp] * 5
            lib.lla_oracle_backward_rows.restype = None
            lib.lla_oracle_gdn_explicit.argtypes = [dp] * 7 + [ctypes.c_int] * 6
            lib.lla_oracle_gdn_explicit.restype = None
            lib.lla_oracle_gdn_recurrent.argtypes = [dp] * 7 + [ctypes.c_int] * 6
            lib.lla_oracle_gdn_recurrent.restype = ctypes.c_int
            lib.lla_oracle_gdn_decode_step.argtypes = [dp] * 7 + [i64p, dp] + [ctypes.c_int] * 5
            lib.lla_oracle_gdn_decode_step.restype = ctypes.c_int
            lib.lla_oracle_gdn_explicit_rows.argtypes = [dp] * 7 + [ctypes.c_int] * 5 + [i64p, ctypes.c_int]
            lib.lla_oracle_gdn_explicit_rows.restype = None
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def level(t: int, s: int) -> int:
    """Fenwick level of key ``s`` for query ``t`` (-1 if ``s > t``)."""
    return int(_load().lla_oracle_level(int(t), int(s)))


def num_levels(T: int) -> int:
    """Number of Fenwick levels reached by a length-``T`` sequence (enumerated)."""
    return int(_load().lla_oracle_num_levels(int(T)))


def _check_forward(q, k, v, log_a, lam):
    q, k, v, log_a, lam = (_f64(x) for x in (q, k, v, log_a, lam))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    L = lam.shape[-1]
    assert k.shape == (B, H, T, dk) and v.shape == (B, H, T, dv)
    assert log_a.shape == (B, H, T) and lam.shape == (B, H, T, L)
    return q, k, v, log_a, lam, (B, H, T, dk, dv, L)


def explicit(q, k, v, log_a, lam) -> np.ndarray:
    """O(T^2) explicit-mask form: (Q K^T (.) M^S (.) M^H) V, fp64."""
    q, k, v, log_a, lam, (B, H, T, dk, dv, L) = _check_forward(q, k, v, log_a, lam)
    out = np.zeros((B, H, T, dv), dtype=np.float64)
    _load().lla_oracle_explicit(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(lam), _ptr(out),
                                B, H, T, dk, dv, L)
    return out


def explicit_rows(q, k, v, log_a, lam, b: int, h: int, rows) -> np.ndarray:
    """Explicit form for chosen query rows of head (b, h) only: returns [len(rows), dv]."""
    sl = (slice(b, b + 1), slice(h, h + 1))
    q, k, v, log_a, lam, (_, _, T, dk, dv, L) = _check_forward(q[sl], k[sl], v[sl], log_a[sl], lam[sl])
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    assert rows.ndim == 1 and (rows >= 0).all() and (rows < T).all()
    out = np.zeros((rows.size, dv), dtype=np.float64)
    _load().lla_oracle_explicit_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(lam), _ptr(out),
                                     0, T, dk, dv, L,
                                     rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), int(rows.size))
    return out


def backward(q, k, v, log_a, lam, dout):
    """Gradients of L = sum(dout * O) for the explicit form, fp64:
    returns (dq, dk, dv, dlog_a, dlambda) with the shapes of (q, k, v, log_a, lambda)."""
    q, k, v, log_a, lam, (B, H, T, dk, dv, L) = _check_forward(q, k, v, log_a, lam)
    dout = _f64(dout)
    assert dout.shape == (B, H, T, dv)
    dq = np.zeros_like(q)
    dk_ = np.zeros_like(k)
    dv_ = np.zeros_like(v)
    dla = np.zeros_like(log_a)
    dlam = np.zeros_like(lam)
    _load().lla_oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(lam), _ptr(dout),
                                _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dla), _ptr(dlam), B, H, T, dk, dv, L)
    return dq, dk_, dv_, dla, dlam


def backward_rows(q, k, v, log_a, lam, dout, b: int, h: int, rows):
    """Backward at chosen positions x of head (b, h): returns (dq [n,dk], dk [n,dk], dv [n,dv],
    dlambda [n,L], dcum [n]) where dcum_x = dlog_a_x - dlog_a_{x+1} (dlog_a_T = 0)."""
    sl = (slice(b, b + 1), slice(h, h + 1))
    q, k, v, log_a, lam, (_, _, T, dk, dv, L) = _check_forward(q[sl], k[sl], v[sl], log_a[sl], lam[sl])
    dout = _f64(dout[sl])
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    assert rows.ndim == 1 and (rows >= 0).all() and (rows < T).all()
    n = rows.size
    out = [np.zeros((n, dk)), np.zeros((n, dk)), np.zeros((n, dv)), np.zeros((n, L)), np.zeros(n)]
    _load().lla_oracle_backward_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(lam), _ptr(dout), 0, T, dk, dv, L,
                                     rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), int(n),
                                     *[_ptr(o) for o in out])
    return tuple(out)


def recurrent(q, k, v, log_a, lam) -> np.ndarray:
    """Token-by-token Fenwick recurrence with lowbit-carry merges, fp64."""
    q, k, v, log_a, lam, (B, H, T, dk, dv, L) = _check_forward(q, k, v, log_a, lam)
    out = np.zeros((B, H, T, dv), dtype=np.float64)
    rc = _load().lla_oracle_recurrent(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(lam), _ptr(out),
                                      B, H, T, dk, dv, L)
    if rc != 0:
        raise MemoryError("oracle state allocation failed")
    return out


def decode_step(q, k, v, log_a, lam, states, t):
    """One recurrent decode step for a batch, fp64.

    ``states`` [B,H,Lmax,dk,dv] is updated in place (it must be a C-contiguous
    float64 array); returns ``out`` [B,H,dv]."""
    q, k, v, log_a, lam = (_f64(x) for x in (q, k, v, log_a, lam))
    assert isinstance(states, np.ndarray) and states.dtype == np.float64 and states.flags.c_contiguous
    t = np.ascontiguousarray(np.asarray(t, dtype=np.int64))
    B, H, dk = q.shape
    dv = v.shape[-1]
    Lmax = states.shape[2]
    assert states.shape == (B, H, Lmax, dk, dv) and lam.shape == (B, H, Lmax) and t.shape == (B,)
    out = np.zeros((B, H, dv), dtype=np.float64)
    rc = _load().lla_oracle_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(lam), _ptr(states),
                                        t.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _ptr(out),
                                        B, H, dk, dv, Lmax)
    if rc != 0:
        raise ValueError("decode position needs more levels than the state set holds")
    return out


# ----------------------------------------------------------------------------- Gated DeltaNet

def _check_gdn(q, k, v, log_a, beta, lam):
    q, k, v, log_a, lam, dims = _check_forward(q, k, v, log_a, lam)
    beta = _f64(beta)
    assert beta.shape == log_a.shape
    return q, k, v, log_a, beta, lam, dims


def gdn_explicit(q, k, v, log_a, beta, lam) -> np.ndarray:
    """Log-linear Gated DeltaNet, explicit O(T^2) form: o_t = sum_{s<=t} lambda_t^(l(t,s)) A[t,s] v_s with
    A[t,s] = beta_s k_s^T A_{s+1} ... A_t q_t and A_r = exp(log_a_r) (I - beta_r k_r k_r^T); fp64."""
    q, k, v, log_a, beta, lam, (B, H, T, dk, dv, L) = _check_gdn(q, k, v, log_a, beta, lam)
    out = np.zeros((B, H, T, dv), dtype=np.float64)
    _load().lla_oracle_gdn_explicit(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(beta), _ptr(lam), _ptr(out),
                                    B, H, T, dk, dv, L)
    return out


def gdn_recurrent(q, k, v, log_a, beta, lam) -> np.ndarray:
    """Log-linear Gated DeltaNet, token-by-token Fenwick recurrence (every held bucket evolves under
    the gated delta-rule transition, lowbit-carry merges); fp64."""
    q, k, v, log_a, beta, lam, (B, H, T, dk, dv, L) = _check_gdn(q, k, v, log_a, beta, lam)
    out = np.zeros((B, H, T, dv), dtype=np.float64)
    rc = _load().lla_oracle_gdn_recurrent(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(beta), _ptr(lam),
                                          _ptr(out), B, H, T, dk, dv, L)
    if rc != 0:
        raise MemoryError("oracle state allocation failed")
    return out


def gdn_decode_step(q, k, v, log_a, beta, lam, states, t):
    """One log-linear Gated DeltaNet decode step for a batch, fp64; ``states`` [B,H,Lmax,dk,dv]
    (C-contiguous float64) is updated in place; returns ``out`` [B,H,dv]."""
    q, k, v, log_a, beta, lam = (_f64(x) for x in (q, k, v, log_a, beta, lam))
    assert isinstance(states, np.ndarray) and states.dtype == np.float64 and states.flags.c_contiguous
    t = np.ascontiguousarray(np.asarray(t, dtype=np.int64))
    B, H, dk = q.shape
    dv = v.shape[-1]
    Lmax = states.shape[2]
    assert states.shape == (B, H, Lmax, dk, dv) and lam.shape == (B, H, Lmax) and t.shape == (B,)
    assert beta.shape == (B, H) and log_a.shape == (B, H)
    out = np.zeros((B, H, dv), dtype=np.float64)
    rc = _load().lla_oracle_gdn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(beta), _ptr(lam),
                                            _ptr(states), t.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                            _ptr(out), B, H, dk, dv, Lmax)
    if rc != 0:
        raise ValueError("decode position needs more levels than the state set holds")
    return out


def gdn_explicit_rows(q, k, v, log_a, beta, lam, b: int, h: int, rows) -> np.ndarray:
    """gdn_explicit for chosen query rows of head (b, h) only: returns [len(rows), dv]."""
    sl = (slice(b, b + 1), slice(h, h + 1))
    q, k, v, log_a, beta, lam, (_, _, T, dk, dv, L) = _check_gdn(q[sl], k[sl], v[sl], log_a[sl], beta[sl], lam[sl])
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    assert rows.ndim == 1 and (rows >= 0).all() and (rows < T).all()
    out = np.zeros((rows.size, dv), dtype=np.float64)
    _load().lla_oracle_gdn_explicit_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(beta), _ptr(lam), _ptr(out),
                                         0, T, dk, dv, L,
                                         rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), int(rows.size))
    return out
