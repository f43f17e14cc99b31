"""ctypes front end of the fp64 CPU oracle (oracle/path_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and bench.py's CPU
baseline / reference arm.  The CUDA library never imports or links it, and it never imports
the CUDA library.

All arrays are numpy float64, C-contiguous.  Heads are flattened: q,k,v,w,dO [n,L,d],
beta/log_f [n,L].
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "path_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

_lib = None
_P = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP).  Returns the library path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        i, d = ctypes.c_int, ctypes.c_double
        _lib.oracle_num_threads.restype = i
        _lib.oracle_fwd_head_rows.argtypes = [i, i, _P, _P, _P, _P, _P, _P, d, i,
                                              ctypes.POINTER(ctypes.c_int), _P, _P]
        _lib.oracle_fwd.argtypes = [i, i, i, _P, _P, _P, _P, _P, _P, d, _P, _P]
        _lib.oracle_logits.argtypes = [i, i, _P, _P, _P, _P, _P, d, _P]
        _lib.oracle_bwd_head.argtypes = [i, i, _P, _P, _P, _P, _P, _P, d, _P, _P, _P, _P, _P, _P, _P]
        _lib.oracle_decode_step.argtypes = [i, i, i, i, _P, _P, _P, _P, _P, _P, _P, d, _P, _P]
        _lib.oracle_prefill_cache.argtypes = [i, i, i, i, _P, _P, _P, _P, _P, _P]
        _lib.oracle_transport_keys.argtypes = [i, i, i, i, ctypes.POINTER(ctypes.c_int), _P, _P, _P, _P]
        _lib.oracle_decode_step_fox.argtypes = [i, i, i, i, _P, _P, _P, _P, _P, _P, _P, _P, _P, d, _P, _P]
        for f in ("oracle_fwd_head_rows", "oracle_fwd", "oracle_logits", "oracle_bwd_head",
                  "oracle_decode_step", "oracle_prefill_cache", "oracle_transport_keys",
                  "oracle_decode_step_fox"):
            getattr(_lib, f).restype = i
    return _lib


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_P)


def _check(rc):
    if rc != 0:
        raise RuntimeError(f"oracle returned {rc}")


def fwd(q, k, v, w, beta, log_f=None, scale=1.0):
    """o [n,L,d], lse [n,L] for heads [n,L,d]."""
    q, k, v, w, beta, log_f = map(_f64, (q, k, v, w, beta, log_f))
    n, L, d = q.shape
    o = np.zeros((n, L, d))
    lse = np.zeros((n, L))
    _check(lib().oracle_fwd(n, L, d, _ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta),
                            _ptr(log_f), float(scale), _ptr(o), _ptr(lse)))
    return o, lse


def fwd_rows(q, k, v, w, beta, log_f, scale, rows):
    """Selected rows of ONE head: q,k,v,w [L,d]; returns o [len(rows),d], lse [len(rows)]."""
    q, k, v, w, beta, log_f = map(_f64, (q, k, v, w, beta, log_f))
    L, d = q.shape
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    o = np.zeros((len(rows), d))
    lse = np.zeros(len(rows))
    _check(lib().oracle_fwd_head_rows(L, d, _ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta),
                                      _ptr(log_f), float(scale), len(rows),
                                      rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                      _ptr(o), _ptr(lse)))
    return o, lse


def logits(q, k, w, beta, log_f=None, scale=1.0):
    """Full logit matrix [L,L] of ONE head (-inf above the diagonal)."""
    q, k, w, beta, log_f = map(_f64, (q, k, w, beta, log_f))
    L, d = q.shape
    S = np.zeros((L, L))
    _check(lib().oracle_logits(L, d, _ptr(q), _ptr(k), _ptr(w), _ptr(beta), _ptr(log_f),
                               float(scale), _ptr(S)))
    return S


def bwd(q, k, v, w, beta, log_f, scale, dO, want_dlogf=False):
    """Gradients for heads [n,L,d]: dict dq,dk,dv,dw [n,L,d], dbeta [n,L] (+ dlog_f)."""
    q, k, v, w, beta, log_f, dO = map(_f64, (q, k, v, w, beta, log_f, dO))
    n, L, d = q.shape
    out = {key: np.zeros((n, L, d)) for key in ("dq", "dk", "dv", "dw")}
    out["dbeta"] = np.zeros((n, L))
    if want_dlogf:
        out["dlog_f"] = np.zeros((n, L))
    for h in range(n):
        _check(lib().oracle_bwd_head(
            L, d, _ptr(q[h]), _ptr(k[h]), _ptr(v[h]), _ptr(w[h]), _ptr(beta[h]),
            None if log_f is None else _ptr(log_f[h]), float(scale), _ptr(dO[h]),
            _ptr(out["dq"][h]), _ptr(out["dk"][h]), _ptr(out["dv"][h]), _ptr(out["dw"][h]),
            _ptr(out["dbeta"][h]), _ptr(out["dlog_f"][h]) if want_dlogf else None))
    return out


def decode_step(k_cache, v_cache, t, q_t, k_t, v_t, w_t, beta_t, scale=1.0, want_lse=False):
    """One decode step, in place on the fp64 caches [n,cap,d]; returns o_t [n,d] (and lse)."""
    assert k_cache.dtype == np.float64 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.float64 and v_cache.flags.c_contiguous
    q_t, k_t, v_t, w_t, beta_t = map(_f64, (q_t, k_t, v_t, w_t, beta_t))
    n, cap, d = k_cache.shape
    o = np.zeros((n, d))
    lse = np.zeros(n) if want_lse else None
    _check(lib().oracle_decode_step(n, d, cap, int(t), _ptr(k_cache), _ptr(v_cache), _ptr(q_t),
                                    _ptr(k_t), _ptr(v_t), _ptr(w_t), _ptr(beta_t), float(scale),
                                    _ptr(o), _ptr(lse)))
    return (o, lse) if want_lse else o


def prefill_cache(k, v, w, beta, cap):
    """Prefill -> decode hand-off: fp64 caches [n,cap,d] holding the L prompt tokens after the
    decode rewrite of every prompt position (row j = H_{L-1}...H_{j+1} k_j, rows >= L zero)."""
    k, v, w, beta = map(_f64, (k, v, w, beta))
    n, L, d = k.shape
    kc = np.zeros((n, cap, d))
    vc = np.zeros((n, cap, d))
    _check(lib().oracle_prefill_cache(n, d, int(cap), L, _ptr(kc), _ptr(vc), _ptr(k), _ptr(v),
                                      _ptr(w), _ptr(beta)))
    return kc, vc


def transport_keys(k, w, beta, rows):
    """Rows of the prefill hand-off one key at a time: [n, len(rows), d] with entry (h, r) equal
    to H_{L-1}...H_{j+1} k_j of head h, j = rows[r] (O((L - j) d) per row)."""
    k, w, beta = map(_f64, (k, w, beta))
    n, L, d = k.shape
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    out = np.zeros((n, len(rows), d))
    _check(lib().oracle_transport_keys(n, d, L, len(rows), rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                       _ptr(k), _ptr(w), _ptr(beta), _ptr(out)))
    return out


def decode_step_fox(k_cache, v_cache, a_cache, t, q_t, k_t, v_t, w_t, beta_t, logf_t, scale=1.0, want_lse=False):
    """One PaTH-FoX decode step, in place on the fp64 caches [n,cap,d] and the prefix cache a [n,cap]
    (a_j = sum_{s<=j} log f_s); returns o_t [n,d] (and lse)."""
    for c in (k_cache, v_cache, a_cache):
        assert c.dtype == np.float64 and c.flags.c_contiguous
    q_t, k_t, v_t, w_t, beta_t, logf_t = map(_f64, (q_t, k_t, v_t, w_t, beta_t, logf_t))
    n, cap, d = k_cache.shape
    o = np.zeros((n, d))
    lse = np.zeros(n) if want_lse else None
    _check(lib().oracle_decode_step_fox(n, d, cap, int(t), _ptr(k_cache), _ptr(v_cache), _ptr(a_cache), _ptr(q_t),
                                        _ptr(k_t), _ptr(v_t), _ptr(w_t), _ptr(beta_t), _ptr(logf_t), float(scale),
                                        _ptr(o), _ptr(lse)))
    return (o, lse) if want_lse else o
