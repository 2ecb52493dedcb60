"""Oracle: the chunked form of the gated delta rule, float64, stage by stage.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; the
tests, the smoke check and the benchmark's CPU-baseline leg do.  It shares no
code with the CUDA path.

It follows the three stages of the chunked method, written out plainly with
numpy (matrix products via einsum/matmul, the triangular inverse by row-by-row
forward substitution), batched over (batch, chunk, head) only:

  stage 0, gate cumsum   G = inclusive cumsum of the natural-log gate g inside
                         each chunk, restarting every C tokens (the chunk-local
                         cumsum of "kernel_fun/kda/_kernels/bwd_scan.py", host
                         wrapper: g2 is that cumsum divided by ln 2; here we stay
                         in base e, so no division).
  stage 1, WY prepare    ("Reuse P as beta tiles in gated deltanet fused prepare":
                         A_g, its inverse, w = A_g^{-1} k_beta, u = A_g^{-1} v_beta)
                         A_ij = beta_i sum_d k_id k_jd exp(G_id - G_jd) for i > j, else 0
                         Tinv = (I + A)^{-1}
                         w = Tinv (k * beta * exp(G)),  u = Tinv (v * beta)
  stage 2, state scan    ("bwd_scan.py" module docstring: hck[c] = h; v' = u - w h;
                         h = exp2(gd) h + kg^T v' with kg = k exp2(G_last - g2))
                         ckpt[c] = h;  v'_c = u_c - w_c h
                         h <- exp(G_last) * h + (k * exp(G_last - G))^T v'_c
  stage 3, chunk output  o = scale [ (q * exp(G)) ckpt[c] + tril_0(Q~) v'_c ],
                         Q~_ij = sum_d q_id k_jd exp(G_id - G_jd) (diagonal included)

For the scalar gate ("GDN") G is one number per (token, head) and broadcasts
over the key dim; for the per-key-dim gate ("KDA") it is a K-vector.

Reading of the pages where they are silent or disagree: the prepare page writes
k_beta = k * beta with no exp(G) and leaves the construction of A_g out.  Only
w = Tinv (k * beta * exp(G)) makes v' = u - w h equal to the token recurrence's
delta, so that form is used (the page's fragment is not followed there).

A sequence whose length T is not a multiple of C ends in a partial chunk.  It
is handled as if padded with tokens that have beta = 0, g = 0 and zero q, k, v:
such a token leaves the state unchanged (S_t = exp(0) S_{t-1} + 0), so the
padding changes no result; outputs are cut back to T tokens and the partial
chunk has its checkpoint like any other (NT = ceil(T / C)).  In the chunked
cumulative gate a padded token repeats the last real value (the cumsum of a
zero g), which keeps every exp(G_i - G_j) bounded.

Grouped value heads: q and k may have fewer heads (H) than the value-side
tensors (HV = G H: v, g, beta, w, u, v', o, the states).  Value head hv then
reads the q and k of head hv // G, the plain meaning of a group sharing its
queries and keys; every stage expands q and k to HV heads that way before it
computes.  (The scan page indexes its tensors by value head, kv heads shared.)

Layouts follow the library boundary (head dim last):
  q, k [B,T,H,K]; w [B,T,HV,K]; v, u, v_new, o [B,T,HV,V]; g, G [B,T,HV] or
  [B,T,HV,K]; beta [B,T,HV]; h0, h_final [B,HV,K,V]; ckpt [B,NT,HV,K,V].
All arrays are numpy float64.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # a torch tensor: read the exact (possibly rounded) values
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _to_chunks(x, C):
    """[B,T,H,...] -> [B,NT,H,C,...] (a view change only)."""
    B, T, H = x.shape[:3]
    rest = x.shape[3:]
    y = x.reshape(B, T // C, C, H, *rest)
    return np.moveaxis(y, 3, 2)


def _from_chunks(y):
    """[B,NT,H,C,...] -> [B,T,H,...]."""
    B, NT, H, C = y.shape[:4]
    rest = y.shape[4:]
    return np.moveaxis(y, 2, 3).reshape(B, NT * C, H, *rest)


def _pad_tokens(x, C, edge=False):
    """Pad [B,T,...] along the token axis to a multiple of C: zeros, or copies of the last token."""
    T = x.shape[1]
    pad = -T % C
    if pad == 0:
        return x
    fill = np.repeat(x[:, -1:], pad, axis=1) if edge else np.zeros((x.shape[0], pad) + x.shape[2:])
    return np.concatenate([x, fill], axis=1)


def _ragged(T, C):
    return T % C != 0


def _expand_heads(x, HV):
    """q or k of H heads as read by HV = G H value heads: value head hv reads head hv // G."""
    x = _f64(x)
    H = x.shape[2]
    if H == HV:
        return x
    if HV % H:
        raise ValueError("the value heads must be a multiple of the q/k heads")
    return np.repeat(x, HV // H, axis=2)


def _gate_vec(G, C):
    """Chunked gate with a trailing key axis: [B,NT,H,C,1] (scalar) or [B,NT,H,C,K]."""
    Gc = _to_chunks(G, C)
    return Gc[..., None] if G.ndim == 3 else Gc


def chunk_cumsum(g, C):
    """Stage 0: G[t] = sum of g[s] for s from the start of t's chunk up to t (inclusive)."""
    g = _f64(g)
    B, T = g.shape[:2]
    if _ragged(T, C):
        return chunk_cumsum(_pad_tokens(g, C), C)[:, :T]
    gc = g.reshape(B, T // C, C, *g.shape[2:])
    return np.cumsum(gc, axis=2).reshape(g.shape)


def forward_substitution_inverse(A):
    """(I + A)^{-1} for strictly lower-triangular A (batched over leading axes).

    Row i of X = (I + A)^{-1} solves X_i + sum_{j<i} A_ij X_j = e_i, so
    X_i = e_i - sum_{j<i} A_ij X_j, taken in order i = 0, 1, ...
    """
    C = A.shape[-1]
    X = np.zeros_like(A)
    for i in range(C):
        row = np.zeros(A.shape[:-2] + (C,))
        row[..., i] = 1.0
        if i:
            row -= np.einsum("...j,...jc->...c", A[..., i, :i], X[..., :i, :])
        X[..., i, :] = row
    return X


def gated_A(k, beta, G, C):
    """A_ij = beta_i sum_d k_id k_jd exp(G_id - G_jd) for i > j, zero elsewhere.

    Returned chunked: [B,NT,H,C,C]."""
    k = _expand_heads(k, _f64(beta).shape[2])
    if _ragged(k.shape[1], C):
        return gated_A(_pad_tokens(_f64(k), C), _pad_tokens(_f64(beta), C), _pad_tokens(_f64(G), C, edge=True), C)
    kc = _to_chunks(_f64(k), C)                 # [B,NT,H,C,K]
    bc = _to_chunks(_f64(beta), C)              # [B,NT,H,C]
    Gc = _gate_vec(_f64(G), C)                  # [B,NT,H,C,1|K]
    A = np.zeros(kc.shape[:-1] + (C,))
    for i in range(1, C):
        # row i against all earlier rows j < i
        gate = np.exp(Gc[..., i:i + 1, :] - Gc[..., :i, :])          # [...,i,1|K]
        A[..., i, :i] = bc[..., i:i + 1] * np.einsum(
            "...d,...jd->...j", kc[..., i, :], kc[..., :i, :] * gate)
    return A


def prepare_wy(k, v, g, beta, C):
    """Stage 0 + 1.  Returns dict(G, A, Tinv, w, u); G/w/u in boundary layout,
    A and Tinv chunked [B,NT,H,C,C]."""
    k, v, beta = _expand_heads(k, _f64(beta).shape[2]), _f64(v), _f64(beta)
    T = k.shape[1]
    if _ragged(T, C):
        p = prepare_wy(_pad_tokens(k, C), _pad_tokens(v, C), _pad_tokens(_f64(g), C), _pad_tokens(beta, C), C)
        return dict(p, G=p["G"][:, :T], w=p["w"][:, :T], u=p["u"][:, :T])
    G = chunk_cumsum(g, C)
    A = gated_A(k, beta, G, C)
    Tinv = forward_substitution_inverse(A)
    kc, vc = _to_chunks(k, C), _to_chunks(v, C)
    bc = _to_chunks(beta, C)[..., None]
    Gc = _gate_vec(G, C)
    k_beta_g = kc * bc * np.exp(Gc)
    v_beta = vc * bc
    w = Tinv @ k_beta_g
    u = Tinv @ v_beta
    return dict(G=G, A=A, Tinv=Tinv, w=_from_chunks(w), u=_from_chunks(u))


def scan_h(k, w, u, G, h0, C):
    """Stage 2: the serial inter-chunk state scan.

    Returns dict(ckpt [B,NT,H,K,V], v_new [B,T,H,V], h_final [B,H,K,V])."""
    k, w, u, G = _expand_heads(k, _f64(w).shape[2]), _f64(w), _f64(u), _f64(G)
    if _ragged(k.shape[1], C):
        T = k.shape[1]
        s = scan_h(_pad_tokens(k, C), _pad_tokens(w, C), _pad_tokens(u, C), _pad_tokens(G, C, edge=True), h0, C)
        return dict(s, v_new=s["v_new"][:, :T])
    B, T, H, K = k.shape
    V = u.shape[-1]
    NT = T // C
    kc, wc, uc = _to_chunks(k, C), _to_chunks(w, C), _to_chunks(u, C)
    Gc = _gate_vec(G, C)                                  # [B,NT,H,C,1|K]
    h = np.zeros((B, H, K, V)) if h0 is None else _f64(h0).copy()
    ckpt = np.zeros((B, NT, H, K, V))
    v_new = np.zeros((B, NT, H, C, V))
    for c in range(NT):
        ckpt[:, c] = h
        vp = uc[:, c] - wc[:, c] @ h                       # [B,H,C,V]
        v_new[:, c] = vp
        G_last = Gc[:, c, :, C - 1, :]                     # [B,H,1|K]
        kg = kc[:, c] * np.exp(G_last[:, :, None, :] - Gc[:, c])   # [B,H,C,K]
        h = np.exp(G_last)[..., None] * h + np.swapaxes(kg, -1, -2) @ vp
    return dict(ckpt=ckpt, v_new=_from_chunks(v_new), h_final=h)


def gated_causal_scores(q, k, G, C):
    """tril_0(Q~) per chunk, Q~_ij = sum_d q_id k_jd exp(G_id - G_jd), diagonal included.

    Returned chunked: [B,NT,H,C,C]."""
    q, k = _expand_heads(q, _f64(G).shape[2]), _expand_heads(k, _f64(G).shape[2])
    if _ragged(q.shape[1], C):
        return gated_causal_scores(_pad_tokens(_f64(q), C), _pad_tokens(_f64(k), C),
                                   _pad_tokens(_f64(G), C, edge=True), C)
    qc, kc = _to_chunks(_f64(q), C), _to_chunks(_f64(k), C)
    Gc = _gate_vec(_f64(G), C)
    Qt = np.zeros(qc.shape[:-1] + (C,))
    for i in range(C):
        gate = np.exp(Gc[..., i:i + 1, :] - Gc[..., :i + 1, :])    # [...,i+1,1|K]
        Qt[..., i, :i + 1] = np.einsum("...d,...jd->...j", qc[..., i, :], kc[..., :i + 1, :] * gate)
    return Qt


def chunk_output(q, k, v_new, ckpt, G, C, scale):
    """Stage 3: o = scale [ (q exp(G)) ckpt[c] + tril_0(Q~) v'_c ]."""
    HV = _f64(v_new).shape[2]
    q, k, v_new, ckpt, G = _expand_heads(q, HV), _expand_heads(k, HV), _f64(v_new), _f64(ckpt), _f64(G)
    if _ragged(q.shape[1], C):
        T = q.shape[1]
        return chunk_output(_pad_tokens(q, C), _pad_tokens(k, C), _pad_tokens(v_new, C), ckpt,
                            _pad_tokens(G, C, edge=True), C, scale)[:, :T]
    qc, vc = _to_chunks(q, C), _to_chunks(v_new, C)
    Gc = _gate_vec(G, C)
    Qt = gated_causal_scores(q, k, G, C)
    inter = (qc * np.exp(Gc)) @ ckpt                       # ckpt [B,NT,H,K,V]
    intra = Qt @ vc
    return _from_chunks(scale * (inter + intra))


def forward_chunked(q, k, v, g, beta, h0, C, scale):
    """All stages.  Returns dict with every intermediate and o, h_final."""
    p = prepare_wy(k, v, g, beta, C)
    s = scan_h(k, p["w"], p["u"], p["G"], h0, C)
    o = chunk_output(q, k, s["v_new"], s["ckpt"], p["G"], C, scale)
    out = dict(p)
    out.update(s)
    out["o"] = o
    return out
