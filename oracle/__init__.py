"""CPU float64 oracle for the chunked gated-delta-rule forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg import this package.  The library and its Python binding never
do, and it shares no code with them (the seeded input generator, which holds no
arithmetic of the method, is the one module both sides use).

Two independent formulations of the forward:
  * `naive_forward`   -- the token-by-token recurrence in plain C (naive_recurrence.c),
                         threaded over (batch, head, block of value columns);
  * `chunked.*`       -- the chunked form stage by stage in numpy (chunked.py),
                         exposing G, A, (I+A)^{-1}, w, u, v', checkpoints, o, h_final.
and two of the backward (the gradient of o and h_final):
  * `naive_backward`  -- reverse mode over the tokens in plain C (naive_adjoint.c);
  * `chunked_backward.*` -- the chunked backward stage by stage in numpy.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import chunked  # noqa: F401
from .chunked import (chunk_cumsum, forward_chunked, forward_substitution_inverse,  # noqa: F401
                      gated_A, prepare_wy, scan_h, chunk_output)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "naive_recurrence.c")
_ADJ_SRC = os.path.join(_HERE, "naive_adjoint.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_naive.so")
_ADJ_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_adjoint.so")
_lib = None
_adj_lib = None
_lock = threading.Lock()


def _compile(src: str, out: str, force: bool) -> str:
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", src, "-o", tmp, "-lm"])
        os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the C oracles with gcc (portable flags: no -march, no FMA contraction)."""
    _compile(_ADJ_SRC, _ADJ_LIB_PATH, force)
    return _compile(_SRC, _LIB_PATH, force)


def load_library(path: str):
    """ctypes handle on a compiled naive_recurrence.c (the tests also load mutated copies)."""
    lib = ctypes.CDLL(path)
    f = lib.oracle_naive_forward
    i64, dp = ctypes.c_int64, ctypes.POINTER(ctypes.c_double)
    f.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_double,
                  dp, dp, dp, dp, dp, dp, dp, dp, dp, i64, ctypes.c_int]
    f.restype = ctypes.c_int
    return lib


def load_adjoint_library(path: str):
    """ctypes handle on a compiled naive_adjoint.c (the tests also load mutated copies)."""
    lib = ctypes.CDLL(path)
    f = lib.oracle_naive_backward
    i64, dp = ctypes.c_int64, ctypes.POINTER(ctypes.c_double)
    f.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_double] + [dp] * 14 + [ctypes.c_int]
    f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _load_adjoint():
    global _adj_lib
    with _lock:
        if _adj_lib is None:
            build()
            _adj_lib = load_adjoint_library(_ADJ_LIB_PATH)
    return _adj_lib


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def naive_forward(q, k, v, g, beta, h0, C, scale, *, with_ckpt=True, nthreads=None, vblock=None,
                  lib=None):
    """Token recurrence in float64.  Returns dict(o, h_final[, ckpt]) as numpy arrays.

    q and k may have fewer heads than v (grouped value heads): value head hv reads
    the q and k of head hv // (HV / H)."""
    HV = chunked._f64(v).shape[2]
    q, k = chunked._expand_heads(q, HV), chunked._expand_heads(k, HV)
    v, g, beta = (chunked._f64(x) for x in (v, g, beta))
    h0 = chunked._f64(h0)
    B, T, H, K = k.shape
    V = v.shape[-1]
    per_k = 1 if g.ndim == 4 else 0
    o = np.zeros((B, T, H, V))
    hf = np.zeros((B, H, K, V))
    ck = np.zeros((B, -(-T // C), H, K, V)) if with_ckpt else None
    nthreads = host_cores() if nthreads is None else int(nthreads)
    if vblock is None:  # enough work items for every thread
        items_per_vblock = B * H
        nb = max(1, min(V, -(-nthreads // items_per_vblock)))
        vblock = -(-V // nb)
    lib = _load() if lib is None else lib
    rc = lib.oracle_naive_forward(B, T, H, K, V, C, per_k, float(scale),
                                      _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                      _ptr(o), _ptr(hf), _ptr(ck), int(vblock), nthreads)
    if rc != 0:
        raise ValueError("oracle_naive_forward rejected its arguments")
    out = dict(o=o, h_final=hf)
    if with_ckpt:
        out["ckpt"] = ck
    return out


def naive_backward(q, k, v, g, beta, h0, do, dh_final, C, scale, *, nthreads=None, lib=None):
    """Gradients of (o, h_final) by reverse mode over the token recurrence, in float64.

    `do` is the loss gradient with respect to o [B,T,H,V]; `dh_final` with respect
    to h_final [B,H,K,V] (None: zero).  Returns dict(dq, dk, dv, dg, dbeta, dh0).

    With grouped value heads (q, k of fewer heads than v) each value head reads
    its group's q and k, and dq, dk of a shared head sum over the group."""
    HV, Hqk = chunked._f64(v).shape[2], chunked._f64(q).shape[2]
    q, k = chunked._expand_heads(q, HV), chunked._expand_heads(k, HV)
    v, g, beta, do = (chunked._f64(x) for x in (v, g, beta, do))
    h0, dh_final = chunked._f64(h0), chunked._f64(dh_final)
    B, T, H, K = k.shape
    V = v.shape[-1]
    per_k = 1 if g.ndim == 4 else 0
    out = dict(dq=np.zeros((B, T, H, K)), dk=np.zeros((B, T, H, K)), dv=np.zeros((B, T, H, V)),
               dg=np.zeros(g.shape), dbeta=np.zeros((B, T, H)), dh0=np.zeros((B, H, K, V)))
    nthreads = host_cores() if nthreads is None else int(nthreads)
    lib = _load_adjoint() if lib is None else lib
    rc = lib.oracle_naive_backward(B, T, H, K, V, C, per_k, float(scale),
                                   _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(do),
                                   _ptr(dh_final), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                                   _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out["dh0"]), nthreads)
    if rc != 0:
        raise ValueError("oracle_naive_backward rejected its arguments")
    from .chunked_backward import group_sum
    out["dq"], out["dk"] = group_sum(out["dq"], Hqk), group_sum(out["dk"], Hqk)
    return out
