"""Oracle: packed variable-length sequences, float64.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; the
tests do.  It shares no code with the CUDA path.

The pages run equal-length batches only ("kernel_fun/kda/_kernels/bwd_scan.py",
host wrapper: T a whole number of chunks).  A packed batch -- n sequences laid
end to end on one token axis, sequence s holding the rows cu[s] .. cu[s+1]-1 --
is read as n independent problems of the same recurrence: sequence s starts
from its own initial state h0[s], its tokens never see another sequence's, and
its final state is h_final[s].  That is the definition this module writes out:
one token-recurrence oracle call per sequence (naive_forward / naive_backward),
the results placed back at the sequence's rows.  An empty sequence has no
outputs, and its final state is its initial state.

Layouts: packed q, k [total,H,K]; v [total,HV,V]; g [total,HV] or [total,HV,K];
beta [total,HV]; o like v.  Per sequence: h0, h_final, dh_final, dh0 [n,HV,K,V].
"""
from __future__ import annotations

import numpy as np

from . import naive_backward, naive_forward


def _spans(cu):
    cu = [int(x) for x in np.asarray(cu).reshape(-1)]
    if len(cu) < 2 or cu[0] != 0 or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must start at 0 and not decrease")
    return list(zip(cu[:-1], cu[1:]))


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def forward(q, k, v, g, beta, cu, h0, C, scale):
    """o [total,HV,V], h_final [n,HV,K,V] of the packed sequences (h0 None: zero states)."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    spans = _spans(cu)
    n, K = len(spans), k.shape[-1]
    HV, V = v.shape[-2], v.shape[-1]
    h0 = np.zeros((n, HV, K, V)) if h0 is None else _f64(h0)
    o = np.zeros(v.shape)
    hf = np.zeros((n, HV, K, V))
    for s, (a, b) in enumerate(spans):
        if b == a:
            hf[s] = h0[s]
            continue
        r = naive_forward(q[None, a:b], k[None, a:b], v[None, a:b], g[None, a:b], beta[None, a:b], h0[s:s + 1],
                          C, scale, with_ckpt=False)
        o[a:b] = r["o"][0]
        hf[s] = r["h_final"][0]
    return o, hf


def backward(q, k, v, g, beta, cu, h0, do, dh_final, C, scale):
    """dict(dq, dk, dv, dg, dbeta packed like their inputs, dh0 [n,HV,K,V]): the gradient of
    forward's (o, h_final) against do (packed like o) and dh_final (None: zero)."""
    q, k, v, g, beta, do = (_f64(x) for x in (q, k, v, g, beta, do))
    spans = _spans(cu)
    n, K = len(spans), k.shape[-1]
    HV, V = v.shape[-2], v.shape[-1]
    h0 = np.zeros((n, HV, K, V)) if h0 is None else _f64(h0)
    dhf = np.zeros((n, HV, K, V)) if dh_final is None else _f64(dh_final)
    out = dict(dq=np.zeros(q.shape), dk=np.zeros(k.shape), dv=np.zeros(v.shape), dg=np.zeros(g.shape),
               dbeta=np.zeros(beta.shape), dh0=np.zeros((n, HV, K, V)))
    for s, (a, b) in enumerate(spans):
        if b == a:
            out["dh0"][s] = dhf[s]
            continue
        r = naive_backward(q[None, a:b], k[None, a:b], v[None, a:b], g[None, a:b], beta[None, a:b], h0[s:s + 1],
                           do[None, a:b], dhf[s:s + 1], C, scale)
        for name in ("dq", "dk", "dv", "dg", "dbeta"):
            out[name][a:b] = r[name][0]
        out["dh0"][s] = r["dh0"][0]
    return out
