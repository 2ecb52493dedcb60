"""Pins of the segment-map oracle (oracle/segments.py) against other things than itself.

- Stitching the segment maps reproduces the serial scan of oracle.chunked (its
  checkpoints at every segment start and its final state), which runs the
  recurrence chunk by chunk instead of composing matrices.
- With beta = 0 there is no delta step: every map is the decay alone,
  M = diag(exp(sum of g over the segment)) and Z = 0, a closed form in the raw g.
- The reverse stitch (transposed maps, last segment first) reproduces the
  backward oracle's serial reverse scan at every segment end and its dh0.
- One-token chunks with g = 0, beta = 2 and unit keys: a chunk is the textbook
  rank-one delta update S <- (I - 2 k k^T) S + 2 k v^T, so M = I - 2 k k^T, a
  reflection (M M = I, det M = -1), and Z = 2 k v^T.
"""
import numpy as np
import pytest
import torch

from chunked_gated_delta_prepare_gb300.inputs import make_inputs
from oracle import chunked, chunked_backward, segments


def _problem(per_k, B=2, T=128, H=2, HV=None, K=8, V=6, seed=61):
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=torch.float32, with_h0=True, seed=seed)
    d = {n: t.double().numpy() for n, t in x.tensors().items()}
    if HV:   # grouped value heads: HV value-side heads over the H q/k heads
        rng = np.random.default_rng(seed)
        d["v"] = rng.standard_normal((B, T, HV, V))
        d["g"] = np.repeat(d["g"], HV // H, axis=2)
        d["beta"] = np.repeat(d["beta"], HV // H, axis=2)
        d["h0"] = rng.standard_normal((B, HV, K, V)) * 0.1
    d["h0"] = d["h0"] * 20
    return d


@pytest.mark.parametrize("per_k", [False, True])
@pytest.mark.parametrize("C,S", [(16, 2), (16, 4), (32, 4), (8, 16)])
def test_stitched_maps_reproduce_the_serial_scan(per_k, C, S):
    d = _problem(per_k)
    p = chunked.prepare_wy(d["k"], d["v"], d["g"], d["beta"], C)
    ref = chunked.scan_h(d["k"], p["w"], p["u"], p["G"], d["h0"], C)
    M, Z = segments.segment_maps(d["k"], p["w"], p["u"], p["G"], C, S)
    starts, hf = segments.stitch(M, Z, d["h0"])
    n = (d["k"].shape[1] // C) // S
    scale = np.abs(ref["h_final"]).max()
    for s in range(S):
        assert np.abs(starts[:, s] - ref["ckpt"][:, s * n]).max() <= 1e-11 * scale
    assert np.abs(hf - ref["h_final"]).max() <= 1e-11 * scale


def test_stitched_maps_with_grouped_value_heads():
    d = _problem(False, H=2, HV=4, seed=62)
    p = chunked.prepare_wy(d["k"], d["v"], d["g"], d["beta"], 16)
    ref = chunked.scan_h(d["k"], p["w"], p["u"], p["G"], d["h0"], 16)
    M, Z = segments.segment_maps(d["k"], p["w"], p["u"], p["G"], 16, 4)
    _, hf = segments.stitch(M, Z, d["h0"])
    assert np.abs(hf - ref["h_final"]).max() <= 1e-11 * np.abs(ref["h_final"]).max()


@pytest.mark.parametrize("per_k", [False, True])
def test_no_delta_step_leaves_the_decay(per_k):
    d = _problem(per_k, seed=63)
    beta = np.zeros_like(d["beta"])
    C, S = 16, 4
    p = chunked.prepare_wy(d["k"], d["v"], d["g"], beta, C)
    M, Z = segments.segment_maps(d["k"], p["w"], p["u"], p["G"], C, S)
    B, T, H = d["g"].shape[:3]
    K = d["k"].shape[-1]
    L = T // S
    for s in range(S):
        tot = d["g"][:, s * L:(s + 1) * L].sum(axis=1)                      # [B,H] or [B,H,K]
        diag = np.exp(tot)[..., None] * np.ones(K) if not per_k else np.exp(tot)
        want = np.einsum("bhd,de->bhde", diag, np.eye(K))
        assert np.abs(M[:, s] - want).max() <= 1e-12
    assert np.abs(Z).max() == 0.0


def test_one_token_chunks_are_reflections():
    rng = np.random.default_rng(64)
    B, T, H, K, V = 1, 8, 1, 5, 3
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    g = np.zeros((B, T, H))
    beta = np.full((B, T, H), 2.0)
    p = chunked.prepare_wy(k, v, g, beta, 1)
    M, Z = segments.segment_maps(k, p["w"], p["u"], p["G"], 1, T)
    for t in range(T):
        kk = k[0, t, 0]
        assert np.abs(M[0, t, 0] - (np.eye(K) - 2 * np.outer(kk, kk))).max() <= 1e-14
        assert np.abs(M[0, t, 0] @ M[0, t, 0] - np.eye(K)).max() <= 1e-13
        assert abs(np.linalg.det(M[0, t, 0]) + 1.0) <= 1e-12
        assert np.abs(Z[0, t, 0] - 2 * np.outer(kk, v[0, t, 0])).max() <= 1e-14


@pytest.mark.parametrize("per_k", [False, True])
@pytest.mark.parametrize("C,S", [(16, 4), (8, 8)])
def test_reverse_stitch_reproduces_the_serial_reverse_scan(per_k, C, S):
    d = _problem(per_k, seed=65)
    rng = np.random.default_rng(66)
    B, T, H, K = d["k"].shape
    V = d["v"].shape[-1]
    do = rng.standard_normal((B, T, H, V))
    dhf = rng.standard_normal((B, H, K, V))
    scale = 0.3
    p = chunked.prepare_wy(d["k"], d["v"], d["g"], d["beta"], C)
    dl = chunked_backward.dv_local(d["q"], d["k"], p["G"], do, C, scale)
    ref = chunked_backward.scan_dh(d["q"], d["k"], p["w"], p["G"], do, dl, dhf, C, scale)
    M, _ = segments.segment_maps(d["k"], p["w"], p["u"], p["G"], C, S)
    L = T // S
    zb = np.stack([chunked_backward.scan_dh(d["q"][:, s * L:(s + 1) * L], d["k"][:, s * L:(s + 1) * L],
                                            p["w"][:, s * L:(s + 1) * L], p["G"][:, s * L:(s + 1) * L],
                                            do[:, s * L:(s + 1) * L], dl[:, s * L:(s + 1) * L], None, C,
                                            scale)["dh0"] for s in range(S)], axis=1)
    ends, dh0 = segments.stitch_reverse(M, zb, dhf)
    n = (T // C) // S
    tol = 1e-11 * np.abs(ref["dh0"]).max()
    for s in range(S):
        assert np.abs(ends[:, s] - ref["dh_ckpt"][:, (s + 1) * n - 1]).max() <= tol
    assert np.abs(dh0 - ref["dh0"]).max() <= tol
