"""Oracle: the segment maps of the state scan, float64.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; the
tests do.  It shares no code with the CUDA path.

The state scan of "kernel_fun/kda/_kernels/bwd_scan.py" (module docstring)
takes one chunk as

    v' = u - w h,   h <- exp(G_last) h + kg^T v',   kg = k exp(G_last - G),

which is affine in h:  h <- A_c h + B_c  with

    A_c = diag(exp(G_last)) - kg^T w      [K, K]
    B_c = kg^T u                          [K, V]

(exp(G_last) is one number for the scalar gate, a K-vector on the diagonal for
the per-key-dim gate).  A run of chunks is then one affine map
h_end = M h_start + Z: M is the product of the run's A_c, the latest on the
left, and Z is the state the run leaves when it starts from zero.  Cutting
each sequence into S equal runs ("segments") and stitching their maps,

    h_start[0] = h0,   h_start[s + 1] = M_s h_start[s] + Z_s,
    h_final = M_{S-1} h_start[S-1] + Z_{S-1},

gives every segment's starting state, after which the segments can be scanned
independently.  The pages scan serially and do not split the scan; this is
the plain algebra of the recurrence they state, written out chunk by chunk.

The backward's reverse scan is affine the other way round: per chunk
dh_before = A_c^T dh_after + b_c (with b_c = scale (q e^G)^T do - w^T dv_loc), so
a segment maps the gradient at its end to the one at its start by M^T, the
transpose of its forward map, plus Z_b, the gradient the segment leaves at its
start from a zero gradient at its end.  Stitching from the last segment,

    end[S-1] = dh_final,   end[s-1] = M_s^T end[s] + Zb_s,   dh0 = M_0^T end[0] + Zb_0.

Layouts: k [B,T,H,K] (q/k heads, expanded to the value heads as in
oracle.chunked), w [B,T,HV,K], u [B,T,HV,V], G [B,T,HV] or [B,T,HV,K];
M [B,S,HV,K,K], Z [B,S,HV,K,V], h_start [B,S,HV,K,V].  T must be a multiple
of C and NT = T / C a multiple of S.
"""
from __future__ import annotations

import numpy as np

from . import chunked


def chunk_maps(k, w, u, G, C):
    """(A, Bc): every chunk's affine map, A [B,NT,H,K,K] and Bc [B,NT,H,K,V]."""
    w, u, G = (np.asarray(x, dtype=np.float64) for x in (w, u, G))
    k = chunked._expand_heads(np.asarray(k, dtype=np.float64), w.shape[2])
    B, T, H, K = k.shape
    if T % C:
        raise ValueError("segment maps need whole chunks")
    NT = T // C
    kc = k.reshape(B, NT, C, H, K).transpose(0, 1, 3, 2, 4)           # [B,NT,H,C,K]
    wc = w.reshape(B, NT, C, H, K).transpose(0, 1, 3, 2, 4)
    uc = u.reshape(B, NT, C, H, -1).transpose(0, 1, 3, 2, 4)          # [B,NT,H,C,V]
    if G.ndim == 3:
        Gc = G.reshape(B, NT, C, H).transpose(0, 1, 3, 2)[..., None]   # [B,NT,H,C,1]
    else:
        Gc = G.reshape(B, NT, C, H, K).transpose(0, 1, 3, 2, 4)       # [B,NT,H,C,K]
    G_last = Gc[..., C - 1:C, :]                                       # [B,NT,H,1,1|K]
    kg = kc * np.exp(G_last - Gc)                                      # [B,NT,H,C,K]
    decay = np.broadcast_to(np.exp(G_last[..., 0, :]), (B, NT, H, K))  # [B,NT,H,K]
    A = np.einsum("...d,de->...de", decay, np.eye(K)) - np.swapaxes(kg, -1, -2) @ wc
    Bc = np.swapaxes(kg, -1, -2) @ uc
    return A, Bc


def segment_maps(k, w, u, G, C, S):
    """(M, Z) of each of the S segments: M [B,S,H,K,K], Z [B,S,H,K,V]."""
    A, Bc = chunk_maps(k, w, u, G, C)
    B, NT, H, K, V = Bc.shape
    if NT % S:
        raise ValueError("the segments must split the chunks evenly")
    n = NT // S
    M = np.zeros((B, S, H, K, K))
    Z = np.zeros((B, S, H, K, V))
    for s in range(S):
        m = np.broadcast_to(np.eye(K), (B, H, K, K)).copy()
        z = np.zeros((B, H, K, V))
        for c in range(s * n, (s + 1) * n):
            # one more chunk after the ones folded so far: h -> A_c (m h + z) + B_c
            m = A[:, c] @ m
            z = A[:, c] @ z + Bc[:, c]
        M[:, s], Z[:, s] = m, z
    return M, Z


def stitch(M, Z, h0):
    """(h_start [B,S,H,K,V], h_final [B,H,K,V]) from the segment maps and h0 (None: zero)."""
    M, Z = np.asarray(M, dtype=np.float64), np.asarray(Z, dtype=np.float64)
    B, S, H, K, V = Z.shape
    h = np.zeros((B, H, K, V)) if h0 is None else np.asarray(h0, dtype=np.float64).copy()
    starts = np.zeros((B, S, H, K, V))
    for s in range(S):
        starts[:, s] = h
        h = M[:, s] @ h + Z[:, s]
    return starts, h


def stitch_reverse(M, Zb, dh_final):
    """(ends [B,S,H,K,V], dh0 [B,H,K,V]): the state gradient at the end of every segment and at
    the start of the sequence, from the forward maps M and the backward offsets Zb (dh_final None: zero)."""
    M, Zb = np.asarray(M, dtype=np.float64), np.asarray(Zb, dtype=np.float64)
    B, S, H, K, V = Zb.shape
    e = np.zeros((B, H, K, V)) if dh_final is None else np.asarray(dh_final, dtype=np.float64).copy()
    ends = np.zeros((B, S, H, K, V))
    for s in range(S - 1, -1, -1):
        ends[:, s] = e
        e = np.swapaxes(M[:, s], -1, -2) @ e + Zb[:, s]
    return ends, e
