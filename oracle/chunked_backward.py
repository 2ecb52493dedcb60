"""Oracle: the chunked backward of the gated delta rule, stage by stage, in float64.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU legs use it; the library never does.  It is the per-stage reference for the
CUDA backward, and is itself pinned to the token-by-token reverse mode of
naive_adjoint.c (and that to finite differences and to autograd).

The forward of one chunk, as chunked.py computes it (rows i, j of the chunk;
G the chunk-local cumsum of g; G_L its last row; h the state before the chunk):

    kb = beta k e^G,  vb = beta v
    A  = strict_lower(beta_i sum_d k_id k_jd e^(G_id - G_jd)),  Tinv = (I + A)^-1
    w  = Tinv kb,  u = Tinv vb,  v' = u - w h
    kg = k e^(G_L - G),  h_next = e^(G_L) h + kg^T v'
    o  = scale [ (q e^G) h + tril0(Qt) v' ],  Qt_ij = sum_d q_id k_jd e^(G_id - G_jd)

"kernel_fun/kda/_kernels/bwd_scan.py" (module docstring) gives the first
backward stage: the forward re-scan that rebuilds the checkpoints h and v'
(chunked.scan_h here).  The rest follows by differentiating the lines above;
with do the gradient of o and dh_next that of h_next, per chunk:

  dv_local   dv_loc = scale tril0(Qt)^T do
  scan_dh    serial over chunks from the last:  dh_ckpt[c] = dh_next,
               dv'   = dv_loc + kg dh_next
               dh    = scale (q e^G)^T do + e^(G_L) dh_next - w^T dv'
             and dh0 = dh after the first chunk
  dqkwg      per chunk, with dqg = scale do h^T, dQt = scale tril0(do v'^T), dkg = v' dh_next^T:
               dq = dqg e^G + L(dQt, k)
               dk = R(dQt, q) + dkg e^(G_L - G)
               dw = -dv' h^T
               dG = dqg (q e^G) + q L(dQt, k) - k R(dQt, q) - dkg kg,
               plus on the last row  sum_i dkg_i kg_i + e^(G_L) sum_v (h dh_next)
  wy_backward with Tinv rebuilt from k, beta, G and du = dv':
               dkb = Tinv^T dw,  dvb = Tinv^T du
               dA  = strict_lower(-Tinv^T (dw kb^T + du vb^T) Tinv^T),  Y = beta_i dA_ij
               dk  = beta e^G dkb + L(Y, k) + R(Y, k)
               dv  = beta dvb
               dbeta = sum_d dkb k e^G + sum_v dvb v + sum_j dA_ij M_ij   (A = beta_i M)
               dG  = dkb kb + k L(Y, k) - k R(Y, k)
  dg         the reverse cumsum of dG within each chunk (G_i = sum of g up to i)

where L(X, Y)_i = sum_j X_ij Y_j e^(G_i - G_j) and R(X, Y)_j = sum_i X_ij Y_i e^(G_i - G_j),
elementwise over the key dim.  For a scalar gate every e^G is a scalar per row
and dG is summed over the key dim.

With grouped value heads (q, k of H heads shared by HV = G H value heads, as in
chunked.py) every stage works per value head on q and k expanded to HV heads,
and dq and dk of a shared head are the sums over its group (`group_sum`).

A partial last chunk is padded as in chunked.py (beta = 0, g = 0, zero q, k, v,
do; G repeats its last value).  A padded row's G is a copy of G at row T - 1,
so the gate gradient of the padded rows is added to row T - 1 before the
padding is cut away; the reverse cumsum then gives every real g its gradient.
"""
from __future__ import annotations

import numpy as np

from .chunked import (_expand_heads, _f64, _from_chunks, _gate_vec, _pad_tokens, _ragged, _to_chunks,
                      forward_substitution_inverse, gated_A, gated_causal_scores, prepare_wy, scan_h)


def group_sum(x, H):
    """[B,T,HV,...] per value head -> [B,T,H,...]: the gradient of a head its group shares."""
    x = _f64(x)
    B, T, HV = x.shape[:3]
    if HV == H:
        return x
    return x.reshape(B, T, H, HV // H, *x.shape[3:]).sum(axis=3)


def _last_row_fold(dG, T):
    """[B,Tp,...] -> [B,T,...]: padded rows' gradient added to row T-1 (their G is a copy of it)."""
    out = dG[:, :T].copy()
    out[:, T - 1] += dG[:, T:].sum(axis=1)
    return out


def _pad_all(C, *xs, edge_last=False):
    pads = [_pad_tokens(_f64(x), C) for x in xs[:-1]]
    pads.append(_pad_tokens(_f64(xs[-1]), C, edge=edge_last))
    return pads


def _pairwise(X, Yl, Yr, Gc):
    """L(X, Yl) and R(X, Yr) for X [..,C,C], Yl and Yr [..,C,D], Gc [..,C,1|K]."""
    C = X.shape[-1]
    Lo = np.zeros(X.shape[:-1] + (np.broadcast_shapes(Yl.shape[-1:], Gc.shape[-1:])[0],))
    Ro = np.zeros_like(Lo)
    for i in range(C):
        gate = np.exp(Gc[..., i:i + 1, :] - Gc)                                 # [..,C(j),D]: e^(G_i - G_j)
        Lo[..., i, :] = np.einsum("...j,...jd->...d", X[..., i, :], Yl * gate)
        Ro += X[..., i, :, None] * (Yr[..., i:i + 1, :] * gate)
    return Lo, Ro


def dv_local(q, k, G, do, C, scale):
    """scale tril0(Qt)^T do, per chunk: [B,T,H,V]."""
    q, k = _expand_heads(q, _f64(do).shape[2]), _expand_heads(k, _f64(do).shape[2])
    T = q.shape[1]
    if _ragged(T, C):
        qp, kp, dop, Gp = _pad_all(C, q, k, do, G, edge_last=True)
        return dv_local(qp, kp, Gp, dop, C, scale)[:, :T]
    Qt = gated_causal_scores(q, k, G, C)                                  # [B,NT,H,C,C]
    doc = _to_chunks(_f64(do), C)
    return _from_chunks(scale * np.swapaxes(Qt, -1, -2) @ doc)


def scan_dh(q, k, w, G, do, dv_loc, dh_final, C, scale):
    """Reverse scan.  Returns dict(dh_ckpt [B,NT,H,K,V] (gradient of the state after
    each chunk), dv_new [B,T,H,V] (gradient of v'), dh0 [B,H,K,V])."""
    q, k = _expand_heads(q, _f64(w).shape[2]), _expand_heads(k, _f64(w).shape[2])
    T = q.shape[1]
    if _ragged(T, C):
        qp, kp, wp, dop, dvp, Gp = _pad_all(C, q, k, w, do, dv_loc, G, edge_last=True)
        r = scan_dh(qp, kp, wp, Gp, dop, dvp, dh_final, C, scale)
        return dict(r, dv_new=r["dv_new"][:, :T])
    qc, kc, wc = (_to_chunks(_f64(x), C) for x in (q, k, w))
    doc, dlc = _to_chunks(_f64(do), C), _to_chunks(_f64(dv_loc), C)
    Gc = _gate_vec(_f64(G), C)
    B, NT, H, _, K = qc.shape
    V = doc.shape[-1]
    dh = np.zeros((B, H, K, V)) if dh_final is None else _f64(dh_final).copy()
    dh_ckpt = np.zeros((B, NT, H, K, V))
    dvn = np.zeros_like(doc)
    for c in range(NT - 1, -1, -1):
        G_last = Gc[:, c, :, -1, :]                                         # [B,H,1|K]
        kg = kc[:, c] * np.exp(G_last[:, :, None, :] - Gc[:, c])             # [B,H,C,K]
        dh_ckpt[:, c] = dh
        dvp = dlc[:, c] + kg @ dh
        dvn[:, c] = dvp
        qg = qc[:, c] * np.exp(Gc[:, c])
        dh = (scale * np.swapaxes(qg, -1, -2) @ doc[:, c] + np.exp(G_last)[..., :, None] * dh
              - np.swapaxes(wc[:, c], -1, -2) @ dvp)
    return dict(dh_ckpt=dh_ckpt, dv_new=_from_chunks(dvn), dh0=dh)


def dqkwg(q, k, v_new, w, G, h_ckpt, dh_ckpt, do, dv_new, C, scale):
    """Per-chunk gradients through the output, the state update and v' = u - w h.

    Returns dict(dq, dk, dw) [B,T,H,K] and dG [B,T,H,K] (per key dim, before the
    sum a scalar gate takes); dq and dk per value head."""
    q, k = _expand_heads(q, _f64(w).shape[2]), _expand_heads(k, _f64(w).shape[2])
    T = q.shape[1]
    if _ragged(T, C):
        qp, kp, vp, wp, dop, dvp, Gp = _pad_all(C, q, k, v_new, w, do, dv_new, G, edge_last=True)
        r = dqkwg(qp, kp, vp, wp, Gp, h_ckpt, dh_ckpt, dop, dvp, C, scale)
        return dict(dq=r["dq"][:, :T], dk=r["dk"][:, :T], dw=r["dw"][:, :T], dG=_last_row_fold(r["dG"], T))
    qc, kc, wc = (_to_chunks(_f64(x), C) for x in (q, k, w))
    vpc, doc, dvc = (_to_chunks(_f64(x), C) for x in (v_new, do, dv_new))
    Gc = _gate_vec(_f64(G), C)                                              # [B,NT,H,C,1|K]
    h = _f64(h_ckpt)                                                        # [B,NT,H,K,V]
    dhn = _f64(dh_ckpt)
    hT, dhnT = np.swapaxes(h, -1, -2), np.swapaxes(dhn, -1, -2)
    eG = np.exp(Gc)
    G_L = Gc[..., -1:, :]                                                   # [B,NT,H,1,1|K]
    kg = kc * np.exp(G_L - Gc)
    mask = np.tril(np.ones((C, C)))
    dqg = scale * doc @ hT                                                  # [..,C,K]
    dQt = scale * (doc @ np.swapaxes(vpc, -1, -2)) * mask                   # [..,C,C]
    dkg = vpc @ dhnT                                                        # [..,C,K]
    Lq, Rq = _pairwise(dQt, kc, qc, Gc)
    dq = dqg * eG + Lq
    dk = Rq + dkg * np.exp(G_L - Gc)
    dw = -dvc @ hT
    dG = dqg * qc * eG + qc * Lq - kc * Rq - dkg * kg
    last = (dkg * kg).sum(axis=-2) + np.exp(G_L[..., 0, :]) * (h * dhn).sum(axis=-1)   # [..,K]
    dG[..., -1, :] += last
    return dict(dq=_from_chunks(dq), dk=_from_chunks(dk), dw=_from_chunks(dw), dG=_from_chunks(dG))


def wy_backward(k, v, beta, G, dw, du, C):
    """Gradients through w = Tinv (beta k e^G) and u = Tinv (beta v), with Tinv rebuilt.

    Returns dict(dk [B,T,H,K] per value head, dv [B,T,H,V], dbeta [B,T,H], dG [B,T,H,K])."""
    k = _expand_heads(k, _f64(beta).shape[2])
    T = k.shape[1]
    if _ragged(T, C):
        kp, vp, bp, dwp, dup, Gp = _pad_all(C, k, v, beta, dw, du, G, edge_last=True)
        r = wy_backward(kp, vp, bp, Gp, dwp, dup, C)
        return dict(dk=r["dk"][:, :T], dv=r["dv"][:, :T], dbeta=r["dbeta"][:, :T], dG=_last_row_fold(r["dG"], T))
    k, v, beta, G = _f64(k), _f64(v), _f64(beta), _f64(G)
    kc, vc, bc = _to_chunks(k, C), _to_chunks(v, C), _to_chunks(beta, C)
    dwc, duc = _to_chunks(_f64(dw), C), _to_chunks(_f64(du), C)
    Gc = _gate_vec(G, C)
    eG = np.exp(Gc)
    A = gated_A(k, beta, G, C)
    M = gated_A(k, np.ones_like(beta), G, C)                                # A = beta_i M
    Ti = forward_substitution_inverse(A)
    TiT = np.swapaxes(Ti, -1, -2)
    kb = kc * bc[..., None] * eG
    vb = vc * bc[..., None]
    dkb = TiT @ dwc
    dvb = TiT @ duc
    dT = dwc @ np.swapaxes(kb, -1, -2) + duc @ np.swapaxes(vb, -1, -2)
    dA = np.tril(-TiT @ dT @ TiT, -1)
    Y = dA * bc[..., :, None]
    Lk, Rk = _pairwise(Y, kc, kc, Gc)
    dk = dkb * bc[..., None] * eG + Lk + Rk
    dv = dvb * bc[..., None]
    dbeta = (dkb * kc * eG).sum(-1) + (dvb * vc).sum(-1) + (dA * M).sum(-1)
    dG = dkb * kb + kc * Lk - kc * Rk
    return dict(dk=_from_chunks(dk), dv=_from_chunks(dv), dbeta=_from_chunks(dbeta), dG=_from_chunks(dG))


def reverse_cumsum(dG, C, per_k):
    """dg_s = sum of dG_i over rows i >= s of s's chunk; a scalar gate first sums dG over keys."""
    dG = _f64(dG)
    if not per_k:
        dG = dG.sum(axis=-1, keepdims=True)
    T = dG.shape[1]
    pad = _pad_tokens(dG, C)                   # zero rows: a partial chunk's padding holds no gradient
    B, Tp = pad.shape[:2]
    dc = pad.reshape(B, Tp // C, C, *pad.shape[2:])
    out = np.flip(np.cumsum(np.flip(dc, axis=2), axis=2), axis=2).reshape(pad.shape)[:, :T]
    return out if per_k else out[..., 0]


def backward_chunked(q, k, v, g, beta, h0, do, dh_final, C, scale):
    """All stages.  Returns dict(dq, dk, dv, dg, dbeta, dh0) and every intermediate."""
    per_k = _f64(g).ndim == 4
    Hqk = _f64(q).shape[2]
    p = prepare_wy(k, v, g, beta, C)
    s = scan_h(k, p["w"], p["u"], p["G"], h0, C)
    dl = dv_local(q, k, p["G"], do, C, scale)
    b = scan_dh(q, k, p["w"], p["G"], do, dl, dh_final, C, scale)
    a = dqkwg(q, k, s["v_new"], p["w"], p["G"], s["ckpt"], b["dh_ckpt"], do, b["dv_new"], C, scale)
    y = wy_backward(k, v, beta, p["G"], a["dw"], b["dv_new"], C)
    dG = a["dG"] + y["dG"]
    return dict(G=p["G"], w=p["w"], u=p["u"], v_new=s["v_new"], h_ckpt=s["ckpt"], dv_local=dl,
                dh_ckpt=b["dh_ckpt"], dv_new=b["dv_new"], dw=a["dw"], dG=dG,
                dq=group_sum(a["dq"], Hqk), dk=group_sum(a["dk"] + y["dk"], Hqk), dv=y["dv"], dbeta=y["dbeta"],
                dg=reverse_cumsum(dG, C, per_k), dh0=b["dh0"])
