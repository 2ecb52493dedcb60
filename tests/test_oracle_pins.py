"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks the float64 oracle (both the C token recurrence and the numpy
chunked form) against something independent: a hand-worked example, a closed
form, an invariant of the gated delta rule, a library routine, or an explicit
matrix-product restatement of the recurrence.  No GPU is used.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import chunked
from chunked_gated_delta_prepare_gb300.inputs import make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def small(per_k, *, B=2, T=192, H=3, K=8, V=5, seed=0, h0_scale=10.0):
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=torch.float32, with_h0=True, seed=seed)
    d = {n: t.double().numpy() for n, t in x.tensors().items()}
    d["h0"] = d["h0"] * h0_scale
    return d


def both(d, C, scale, **kw):
    n = oracle.naive_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], C, scale, **kw)
    c = oracle.forward_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], C, scale)
    return n, c


def explicit_matrix_recurrence(d, scale):
    """S_t = (I - beta k k^T) D_t S_{t-1} + beta k v^T with every matrix built explicitly."""
    q, k, v, g, beta, h0 = d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"]
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    hf = np.zeros((B, H, K, V))
    for b in range(B):
        for h in range(H):
            S = h0[b, h].copy() if h0 is not None else np.zeros((K, V))
            for t in range(T):
                kt = k[b, t, h][:, None]
                D = np.diag(np.exp(g[b, t, h])) if g.ndim == 4 else math.exp(g[b, t, h]) * np.eye(K)
                S = (np.eye(K) - beta[b, t, h] * kt @ kt.T) @ D @ S + beta[b, t, h] * kt @ v[b, t, h][None, :]
                o[b, t, h] = scale * S.T @ q[b, t, h]
            hf[b, h] = S
    return o, hf


# ---------------------------------------------------------------- worked examples

def load_golden():
    with open(GOLDEN) as f:
        return json.load(f)["examples"]


@pytest.mark.parametrize("ex", load_golden(), ids=lambda e: e["name"])
@pytest.mark.parametrize("C", [1, 2])
def test_hand_worked_example(ex, C):
    T, K, V = ex["T"], ex["K"], ex["V"]
    q = np.array(ex["q"]).reshape(1, T, 1, K)
    k = np.array(ex["k"]).reshape(1, T, 1, K)
    v = np.array(ex["v"]).reshape(1, T, 1, V)
    gf = np.log(np.array(ex["g_decay_factor"]))
    g = gf.reshape(1, T, 1, K) if ex["gate"] == "per_key_dim" else gf.reshape(1, T, 1)
    beta = np.array(ex["beta"]).reshape(1, T, 1)
    h0 = np.array(ex["h0"]).reshape(1, 1, K, V)
    o_ref = np.array(ex["o"]).reshape(1, T, 1, V)
    h_ref = np.array(ex["h_final"]).reshape(1, 1, K, V)
    n = oracle.naive_forward(q, k, v, g, beta, h0, C, ex["scale"])
    c = oracle.forward_chunked(q, k, v, g, beta, h0, C, ex["scale"])
    for res in (n, c):
        np.testing.assert_allclose(res["o"], o_ref, rtol=0, atol=1e-13)
        np.testing.assert_allclose(res["h_final"], h_ref, rtol=0, atol=1e-13)
    # checkpoint 0 is the initial state
    np.testing.assert_allclose(n["ckpt"][:, 0], h0, atol=0)
    np.testing.assert_allclose(c["ckpt"][:, 0], h0, atol=0)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("per_k", [False, True])
def test_naive_matches_explicit_matrix_products(per_k):
    d = small(per_k, B=1, T=40, H=2, K=6, V=4, seed=3)
    o_ref, h_ref = explicit_matrix_recurrence(d, 0.7)
    n = oracle.naive_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 8, 0.7)
    np.testing.assert_allclose(n["o"], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(n["h_final"], h_ref, rtol=0, atol=1e-12)


def test_single_token_closed_form():
    """T = 1, scalar gate: S_1 = e^g h0 + beta k (v - e^g h0^T k)^T and o = scale S_1^T q."""
    rng = np.random.default_rng(7)
    K, V = 5, 3
    q, k, v = rng.normal(size=K), rng.normal(size=K), rng.normal(size=V)
    g, beta, h0 = -0.3, 0.8, rng.normal(size=(K, V))
    scale = 0.25
    a = math.exp(g)
    S1 = np.empty((K, V))
    for i in range(K):
        for j in range(V):
            r = sum(a * h0[m, j] * k[m] for m in range(K))
            S1[i, j] = a * h0[i, j] + beta * k[i] * (v[j] - r)
    o = [scale * sum(S1[i, j] * q[i] for i in range(K)) for j in range(V)]
    args = (q.reshape(1, 1, 1, K), k.reshape(1, 1, 1, K), v.reshape(1, 1, 1, V),
            np.full((1, 1, 1), g), np.full((1, 1, 1), beta), h0.reshape(1, 1, K, V))
    n = oracle.naive_forward(*args, 1, scale)
    c = oracle.forward_chunked(*args, 1, scale)
    for res in (n, c):
        np.testing.assert_allclose(res["h_final"][0, 0], S1, atol=1e-14)
        np.testing.assert_allclose(res["o"][0, 0, 0], o, atol=1e-14)


# ---------------------------------------------------------------- chunked == naive

@pytest.mark.parametrize("per_k", [False, True])
@pytest.mark.parametrize("C", [16, 32, 64])
def test_chunked_equals_token_recurrence(per_k, C):
    d = small(per_k, seed=C)
    n, c = both(d, C, 0.3)
    for key in ("o", "h_final", "ckpt"):
        assert np.abs(n[key] - c[key]).max() <= 1e-10, key


@pytest.mark.parametrize("per_k", [False, True])
def test_chunk_size_invariance(per_k):
    d = small(per_k, T=128, seed=11)
    outs = [oracle.forward_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], C, 0.5)
            for C in (8, 16, 32, 64, 128)]
    for r in outs[1:]:
        assert np.abs(r["o"] - outs[0]["o"]).max() <= 1e-10
        assert np.abs(r["h_final"] - outs[0]["h_final"]).max() <= 1e-10


# ---------------------------------------------------------------- the inverse

@pytest.mark.parametrize("per_k", [False, True])
def test_inverse_is_exact(per_k):
    d = small(per_k, T=128, K=16, seed=5)
    p = chunked.prepare_wy(d["k"], d["v"], d["g"], d["beta"], 64)
    A, X = p["A"], p["Tinv"]
    eye = np.eye(64)
    assert np.abs(np.triu(A)).max() == 0.0                        # strictly lower
    assert np.abs(X @ (eye + A) - eye).max() <= 1e-12
    assert np.abs((eye + A) @ X - eye).max() <= 1e-12
    np.testing.assert_allclose(X, np.linalg.inv(eye + A), atol=1e-12)  # library routine


def test_gated_A_small_case_by_hand():
    """A_10 = beta_1 (k_1 . k_0) exp(G_1 - G_0) = beta_1 (k_1 . k_0) exp(g_1) for a scalar gate."""
    k = np.array([[1.0, 2.0], [3.0, -1.0]]).reshape(1, 2, 1, 2)
    beta = np.array([0.5, 0.25]).reshape(1, 2, 1)
    g = np.array([-0.1, -0.7]).reshape(1, 2, 1)
    G = chunked.chunk_cumsum(g, 2)
    A = chunked.gated_A(k, beta, G, 2)[0, 0, 0]
    assert A[0, 0] == 0 and A[0, 1] == 0 and A[1, 1] == 0
    assert abs(A[1, 0] - 0.25 * (3 - 2) * math.exp(-0.7)) < 1e-15


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("per_k", [False, True])
def test_beta_zero_decays_initial_state(per_k):
    d = small(per_k, T=96, seed=2)
    d["beta"] = np.zeros_like(d["beta"])
    n, c = both(d, 32, 0.4)
    g = d["g"]
    G_abs = np.cumsum(g, axis=1)                                    # from the sequence start
    if per_k:
        decay = np.exp(G_abs)                                       # [B,T,H,K]
        h_t = decay[..., :, None] * d["h0"][:, None]                # [B,T,H,K,V]
    else:
        h_t = np.exp(G_abs)[..., None, None] * d["h0"][:, None]
    o_ref = 0.4 * np.einsum("bthkv,bthk->bthv", h_t, d["q"])
    for r in (n, c):
        np.testing.assert_allclose(r["h_final"], h_t[:, -1], atol=1e-13)
        np.testing.assert_allclose(r["o"], o_ref, atol=1e-13)
    np.testing.assert_allclose(c["w"], 0.0, atol=0)
    np.testing.assert_allclose(c["u"], 0.0, atol=0)
    np.testing.assert_allclose(c["v_new"], 0.0, atol=0)


def test_beta_zero_no_decay_is_q_h0():
    d = small(False, T=64, seed=4)
    d["beta"][:] = 0.0
    d["g"][:] = 0.0
    n, c = both(d, 16, 0.9)
    o_ref = 0.9 * np.einsum("bhkv,bthk->bthv", d["h0"], d["q"])
    for r in (n, c):
        np.testing.assert_allclose(r["o"], o_ref, atol=1e-13)


@pytest.mark.parametrize("C", [4, 8])
def test_orthonormal_keys_overwrite(C):
    """g = 0, beta = 1, k_t = e_{pi(t)}: the state column read by e_{pi(t)} is v_t (last write wins)."""
    rng = np.random.default_rng(0)
    K, V, T = 8, 3, 16
    pi = np.concatenate([rng.permutation(K), rng.permutation(K)])  # every key written twice
    k = np.zeros((1, T, 1, K))
    k[0, np.arange(T), 0, pi] = 1.0
    q = k.copy()
    v = rng.normal(size=(1, T, 1, V))
    g = np.zeros((1, T, 1))
    beta = np.ones((1, T, 1))
    h0 = rng.normal(size=(1, 1, K, V))
    d = dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0)
    n, c = both(d, C, 1.0)
    for r in (n, c):
        for t in range(T):
            np.testing.assert_allclose(r["o"][0, t, 0], v[0, t, 0], atol=1e-13)  # read right after write
        last = {int(pi[t]): t for t in range(T)}
        for key, t in last.items():
            np.testing.assert_allclose(r["h_final"][0, 0, key], v[0, t, 0], atol=1e-13)


@pytest.mark.parametrize("per_k", [False, True])
def test_strong_decay_forgets(per_k):
    d = small(per_k, T=64, seed=8)
    d["g"] = np.full_like(d["g"], -50.0)
    n, c = both(d, 16, 0.6)
    kq = np.einsum("bthk,bthk->bth", d["k"], d["q"])
    o_ref = 0.6 * (d["beta"] * kq)[..., None] * d["v"]
    h_ref = d["beta"][:, -1, :, None, None] * d["k"][:, -1, :, :, None] * d["v"][:, -1, :, None, :]
    for r in (n, c):
        np.testing.assert_allclose(r["o"], o_ref, atol=1e-12)
        np.testing.assert_allclose(r["h_final"], h_ref, atol=1e-12)


# ---------------------------------------------------------------- invariants

def test_per_key_gate_constant_over_k_equals_scalar_gate():
    d = small(False, T=96, seed=9)
    dk = dict(d)
    dk["g"] = np.repeat(d["g"][..., None], d["k"].shape[-1], axis=-1)
    ns, cs = both(d, 32, 0.5)
    nk, ck = both(dk, 32, 0.5)
    for a, b in ((ns, nk), (cs, ck)):
        np.testing.assert_allclose(a["o"], b["o"], atol=1e-13)
        np.testing.assert_allclose(a["h_final"], b["h_final"], atol=1e-13)


@pytest.mark.parametrize("per_k", [False, True])
def test_state_carry(per_k):
    d = small(per_k, T=128, seed=12)
    full = oracle.naive_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 32, 0.5)
    T1 = 64
    a = {n: (x[:, :T1] if n != "h0" else x) for n, x in d.items()}
    b = {n: x[:, T1:] for n, x in d.items() if n != "h0"}
    for impl in ("naive", "chunked"):
        f = oracle.naive_forward if impl == "naive" else oracle.forward_chunked
        r1 = f(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], 32, 0.5)
        r2 = f(b["q"], b["k"], b["v"], b["g"], b["beta"], r1["h_final"], 32, 0.5)
        np.testing.assert_allclose(np.concatenate([r1["o"], r2["o"]], axis=1), full["o"], atol=1e-12)
        np.testing.assert_allclose(r2["h_final"], full["h_final"], atol=1e-12)


@pytest.mark.parametrize("per_k", [False, True])
def test_linear_in_values_and_initial_state(per_k):
    d1 = small(per_k, T=64, seed=13)
    d2 = small(per_k, T=64, seed=14)
    d2 = dict(d1, v=d2["v"], h0=d2["h0"])
    dm = dict(d1, v=2.0 * d1["v"] - 3.0 * d2["v"], h0=2.0 * d1["h0"] - 3.0 * d2["h0"])
    for f in (oracle.naive_forward, oracle.forward_chunked):
        r1, r2, rm = (f(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], 16, 0.5) for x in (d1, d2, dm))
        np.testing.assert_allclose(rm["o"], 2 * r1["o"] - 3 * r2["o"], atol=1e-12)
        np.testing.assert_allclose(rm["h_final"], 2 * r1["h_final"] - 3 * r2["h_final"], atol=1e-12)


def test_naive_thread_and_block_split_is_exact():
    d = small(True, T=64, V=7, seed=15)
    r1 = oracle.naive_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 16, 0.5, nthreads=1, vblock=7)
    r2 = oracle.naive_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 16, 0.5, nthreads=3, vblock=2)
    for key in ("o", "h_final", "ckpt"):
        assert np.array_equal(r1[key], r2[key])


def test_stage_functions_compose():
    d = small(True, T=64, seed=16)
    full = oracle.forward_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 16, 0.5)
    p = chunked.prepare_wy(d["k"], d["v"], d["g"], d["beta"], 16)
    s = chunked.scan_h(d["k"], p["w"], p["u"], p["G"], d["h0"], 16)
    o = chunked.chunk_output(d["q"], d["k"], s["v_new"], s["ckpt"], p["G"], 16, 0.5)
    assert np.array_equal(o, full["o"])
    np.testing.assert_allclose(p["G"][:, 15], d["g"][:, :16].sum(axis=1), atol=1e-15)
    np.testing.assert_allclose(p["G"][:, 16], d["g"][:, 16], atol=0)   # restarts each chunk


# ---------------------------------------------------------------- a partial last chunk

@pytest.mark.parametrize("per_k", [False, True])
@pytest.mark.parametrize("T,C", [(100, 32), (77, 64), (13, 16), (130, 64)])
def test_partial_last_chunk_matches_explicit_matrices(per_k, T, C):
    # the explicit matrix recurrence knows nothing of chunks, so a ragged tail that the
    # chunked form got wrong (a lost token, a bad cumsum pad, a skipped checkpoint) shows here
    d = small(per_k, T=T, K=6, V=5, seed=T + C)
    eo, ehf = explicit_matrix_recurrence(d, 0.4)
    n, c = both(d, C, 0.4)
    for r in (n, c):
        assert r["o"].shape == (2, T, 3, 5)
        np.testing.assert_allclose(r["o"], eo, atol=1e-11)
        np.testing.assert_allclose(r["h_final"], ehf, atol=1e-11)
    assert n["ckpt"].shape[1] == -(-T // C) and c["ckpt"].shape[1] == -(-T // C)
    assert np.abs(n["ckpt"] - c["ckpt"]).max() <= 1e-11


@pytest.mark.parametrize("per_k", [False, True])
def test_partial_chunk_checkpoint_is_the_prefix_state(per_k):
    # the last (partial) chunk's checkpoint is the state after the whole chunks before it
    T, C = 100, 32
    d = small(per_k, T=T, seed=41)
    full = oracle.naive_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], C, 0.5)
    T1 = (T // C) * C
    pre = {n: (x[:, :T1] if n != "h0" else x) for n, x in d.items()}
    r = oracle.naive_forward(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"], pre["h0"], C, 0.5)
    np.testing.assert_allclose(full["ckpt"][:, -1], r["h_final"], atol=1e-12)
    np.testing.assert_allclose(full["ckpt"][:, :-1], r["ckpt"], atol=1e-12)


@pytest.mark.parametrize("per_k", [False, True])
def test_ragged_chunk_size_invariance(per_k):
    d = small(per_k, T=90, seed=42)
    outs = [oracle.forward_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], C, 0.5)
            for C in (1, 7, 16, 64, 128)]
    for r in outs[1:]:
        assert np.abs(r["o"] - outs[0]["o"]).max() <= 1e-10
        assert np.abs(r["h_final"] - outs[0]["h_final"]).max() <= 1e-10


@pytest.mark.parametrize("per_k", [False, True])
def test_zero_tokens_are_identity_updates(per_k):
    # beta = 0 and g = 0 make S_t = S_{t-1}: appending such tokens leaves h_final as it was
    d = small(per_k, T=40, seed=43)
    r = oracle.naive_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 8, 0.5)
    e = {n: (np.concatenate([x, np.zeros((x.shape[0], 9) + x.shape[2:])], axis=1) if n != "h0" else x)
         for n, x in d.items()}
    e["q"][:, 40:] = 1.0   # any q reads the unchanged state
    re = oracle.naive_forward(e["q"], e["k"], e["v"], e["g"], e["beta"], e["h0"], 8, 0.5)
    np.testing.assert_allclose(re["h_final"], r["h_final"], atol=1e-13)
    np.testing.assert_allclose(re["o"][:, :40], r["o"], atol=1e-13)
    np.testing.assert_allclose(re["o"][:, 40:], 0.5 * np.einsum("bhkv,btk->bthv", r["h_final"],
                                                                np.ones((2, 9, 8))), atol=1e-12)


# ---------------------------------------------------------------- grouped value heads

def grouped(per_k, *, B=2, T=40, H=2, G=3, K=6, V=5, seed=0):
    """q, k with H heads; v, g, beta, h0 with H*G value heads."""
    x = make_inputs(B, T, H * G, K, V, per_k_gate=per_k, io_dtype=torch.float32, with_h0=True, seed=seed)
    d = {n: t.double().numpy() for n, t in x.tensors().items()}
    d["h0"] = d["h0"] * 10.0
    rng = np.random.default_rng(seed)
    d["q"] = rng.standard_normal((B, T, H, K)) / np.sqrt(K)
    d["k"] = rng.standard_normal((B, T, H, K))
    d["k"] /= np.linalg.norm(d["k"], axis=-1, keepdims=True)
    return d


@pytest.mark.parametrize("per_k", [False, True])
def test_grouped_heads_match_a_per_value_head_recurrence(per_k):
    # each value head hv runs the plain recurrence on the q and k of head hv // G (indexed here
    # directly, not through the oracle's expansion), with its own v, g, beta and state
    d = grouped(per_k, seed=51)
    B, T, HV = d["v"].shape[:3]
    H = d["q"].shape[2]
    G = HV // H
    n = oracle.naive_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 16, 0.4)
    c = oracle.forward_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 16, 0.4)
    for hv in range(HV):
        one = dict(q=d["q"][:, :, hv // G: hv // G + 1], k=d["k"][:, :, hv // G: hv // G + 1],
                   v=d["v"][:, :, hv:hv + 1], g=d["g"][:, :, hv:hv + 1], beta=d["beta"][:, :, hv:hv + 1],
                   h0=d["h0"][:, hv:hv + 1])
        eo, eh = explicit_matrix_recurrence(one, 0.4)
        for r in (n, c):
            np.testing.assert_allclose(r["o"][:, :, hv:hv + 1], eo, atol=1e-11)
            np.testing.assert_allclose(r["h_final"][:, hv:hv + 1], eh, atol=1e-11)


def test_grouped_heads_with_equal_value_sides_agree():
    # value heads of one group that share v, g, beta and h0 as well give identical results
    d = grouped(True, H=1, G=2, seed=52)
    for n in ("v", "g", "beta"):
        d[n][:, :, 1] = d[n][:, :, 0]
    d["h0"][:, 1] = d["h0"][:, 0]
    r = oracle.naive_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 8, 0.5)
    assert np.array_equal(r["o"][:, :, 0], r["o"][:, :, 1])
