"""CPU float64 oracle for the chunked gated-delta-rule forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg import this package.  The library and its Python binding never
do, and it shares no code with them (the seeded input generator, which holds no
arithmetic of the method, is the one module both sides use).

Two independent formulations:
  * `naive_forward`   -- the token-by-token recurrence in plain C (naive_recurrence.c),
                         threaded over (batch, head, block of value columns);
  * `chunked.*`       -- the chunked form stage by stage in numpy (chunked.py),
                         exposing G, A, (I+A)^{-1}, w, u, v', checkpoints, o, h_final.
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
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_naive.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags: no -march, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """ctypes handle on a compiled naive_recurrence.c (the tests also load mutated copies)."""
    lib = ctypes.CDLL(path)
    f = lib.oracle_naive_forward
    i64, dp = ctypes.c_int64, ctypes.POINTER(ctypes.c_double)
    f.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_double,
                  dp, dp, dp, dp, dp, dp, dp, dp, dp, i64, ctypes.c_int]
    f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


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
    """Token recurrence in float64.  Returns dict(o, h_final[, ckpt]) as numpy arrays."""
    q, k, v, g, beta = (chunked._f64(x) for x in (q, k, v, g, beta))
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
