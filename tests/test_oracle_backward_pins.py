"""Pins for the backward oracles (oracle/naive_adjoint.c and oracle/chunked_backward.py).

The token-by-token reverse mode is checked against two things that do not share
its derivation: central finite differences of the (separately pinned) forward
oracle, and torch's autograd through an explicit float64 token recurrence.  The
chunked backward is then checked against the token reverse mode, and both
against closed forms that hold when beta = 0.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import chunked_backward as cb
from chunked_gated_delta_prepare_gb300.inputs import make_inputs

GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dh0")
INPUT_OF = dict(dq="q", dk="k", dv="v", dg="g", dbeta="beta", dh0="h0")


def problem(per_k, *, B=2, T=64, H=2, K=6, V=5, seed=0, h0_scale=10.0):
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=torch.float32, with_h0=True, seed=seed)
    d = {n: t.double().numpy() for n, t in x.tensors().items()}
    d["h0"] = d["h0"] * h0_scale
    rng = np.random.default_rng(seed + 1000)
    do = rng.standard_normal((B, T, H, V))
    dhf = rng.standard_normal((B, H, K, V))
    return d, do, dhf


def adjoint(d, do, dhf, C, scale, **kw):
    return oracle.naive_backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], do, dhf, C, scale, **kw)


def rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


# ---------------------------------------------------------------- finite differences

@pytest.mark.parametrize("per_k", [False, True])
def test_adjoint_matches_finite_differences(per_k):
    # central differences of L = sum(do o) + sum(dhf h_final) through the forward oracle
    d, do, dhf = problem(per_k, B=1, T=7, H=1, K=3, V=2, seed=3, h0_scale=30.0)
    scale = 0.7

    def loss():
        r = oracle.naive_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 3, scale, with_ckpt=False)
        return float((r["o"] * do).sum() + (r["h_final"] * dhf).sum())

    got = adjoint(d, do, dhf, 3, scale)
    for name in GRADS:
        x = d[INPUT_OF[name]]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + 1e-6
            lp = loss()
            x[idx] = old - 1e-6
            lm = loss()
            x[idx] = old
            fd[idx] = (lp - lm) / 2e-6
        assert rel(got[name], fd) <= 1e-7, name


# ---------------------------------------------------------------- autograd

def autograd_grads(d, do, dhf, scale):
    t = {n: torch.tensor(x, dtype=torch.float64, requires_grad=True) for n, x in d.items()}
    q, k, v, g, beta, h0 = (t[n] for n in ("q", "k", "v", "g", "beta", "h0"))
    S = h0
    outs = []
    for s in range(k.shape[1]):
        dec = torch.exp(g[:, s])
        St = dec[..., :, None] * S if g.dim() == 4 else dec[..., None, None] * S
        r = v[:, s] - torch.einsum("bhkv,bhk->bhv", St, k[:, s])
        S = St + beta[:, s][..., None, None] * k[:, s][..., :, None] * r[..., None, :]
        outs.append(scale * torch.einsum("bhkv,bhk->bhv", S, q[:, s]))
    loss = (torch.stack(outs, 1) * torch.from_numpy(do)).sum() + (S * torch.from_numpy(dhf)).sum()
    loss.backward()
    return {name: t[INPUT_OF[name]].grad.numpy() for name in GRADS}


@pytest.mark.parametrize("per_k", [False, True])
def test_adjoint_matches_autograd(per_k):
    d, do, dhf = problem(per_k, T=40, seed=5)
    ref = autograd_grads(d, do, dhf, 0.45)
    got = adjoint(d, do, dhf, 16, 0.45)
    for name in GRADS:
        assert rel(got[name], ref[name]) <= 1e-11, name


# ---------------------------------------------------------------- replay and threads

@pytest.mark.parametrize("per_k", [False, True])
def test_adjoint_replay_stretch_changes_nothing(per_k):
    d, do, dhf = problem(per_k, T=50, seed=6)
    runs = [adjoint(d, do, dhf, C, 0.5, nthreads=nt) for C, nt in ((1, 1), (7, 3), (16, 2), (64, 4))]
    for r in runs[1:]:
        for name in GRADS:
            assert np.array_equal(r[name], runs[0][name]), name


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("per_k", [False, True])
def test_beta_zero_no_decay_closed_form(per_k):
    # beta = 0, g = 0: S_t = h0 for every t, o_t = scale h0^T q_t.  With E_t = dhf + scale sum_{s>=t} q_s do_s^T:
    # dq_t = scale h0 do_t, dk = dv = 0, dbeta_t = (v_t - h0^T k_t) . (E_t^T k_t),
    # dg_t = sum of h0 * E_t (per key row, or over all for a scalar gate), dh0 = E_1.
    d, do, dhf = problem(per_k, B=1, T=24, H=1, seed=7)
    d["beta"][:] = 0.0
    d["g"][:] = 0.0
    scale = 0.6
    got = adjoint(d, do, dhf, 8, scale)
    h0, q, k, v = d["h0"][0, 0], d["q"][0, :, 0], d["k"][0, :, 0], d["v"][0, :, 0]
    dO = do[0, :, 0]
    T = q.shape[0]
    E = np.zeros((T + 1,) + h0.shape)
    E[T] = dhf[0, 0]
    for t in range(T - 1, -1, -1):
        E[t] = E[t + 1] + scale * np.outer(q[t], dO[t])
    np.testing.assert_allclose(got["dq"][0, :, 0], scale * dO @ h0.T, atol=1e-12)
    assert np.abs(got["dk"]).max() == 0.0 and np.abs(got["dv"]).max() == 0.0
    dbeta = np.array([(v[t] - h0.T @ k[t]) @ (E[t].T @ k[t]) for t in range(T)])
    np.testing.assert_allclose(got["dbeta"][0, :, 0], dbeta, atol=1e-11)
    dg = np.array([(h0 * E[t]).sum(axis=1) for t in range(T)])
    np.testing.assert_allclose(got["dg"][0, :, 0], dg if per_k else dg.sum(axis=1), atol=1e-11)
    np.testing.assert_allclose(got["dh0"][0, 0], E[0], atol=1e-12)


def test_single_token_closed_form():
    # T = 1, scalar gate: S_1 = a h0 + beta k (v - a h0^T k)^T with a = e^g, o = scale S_1^T q.
    rng = np.random.default_rng(8)
    K, V = 4, 3
    q, k, v, h0, do, dhf = (rng.standard_normal(s) for s in (K, K, V, (K, V), V, (K, V)))
    g, beta, scale = -0.3, 0.8, 0.5
    a = np.exp(g)
    r = v - a * h0.T @ k
    S1 = a * h0 + beta * np.outer(k, r)
    dS = dhf + scale * np.outer(q, do)                      # gradient of S_1
    dd = dS.T @ k                                           # of delta = beta r
    d = dict(q=q[None, None, None], k=k[None, None, None], v=v[None, None, None],
             g=np.array(g).reshape(1, 1, 1), beta=np.array(beta).reshape(1, 1, 1), h0=h0[None, None])
    got = adjoint(d, do[None, None, None], dhf[None, None], 1, scale)
    np.testing.assert_allclose(got["dq"][0, 0, 0], scale * S1 @ do, atol=1e-13)
    np.testing.assert_allclose(got["dv"][0, 0, 0], beta * dd, atol=1e-13)
    np.testing.assert_allclose(got["dk"][0, 0, 0], beta * dS @ r - a * h0 @ (beta * dd), atol=1e-13)
    np.testing.assert_allclose(got["dbeta"][0, 0, 0], r @ dd, atol=1e-13)
    dSt = dS - np.outer(k, beta * dd)
    np.testing.assert_allclose(got["dg"][0, 0, 0], (a * h0 * dSt).sum(), atol=1e-13)
    np.testing.assert_allclose(got["dh0"][0, 0], a * dSt, atol=1e-13)


# ---------------------------------------------------------------- chunked == token reverse mode

@pytest.mark.parametrize("per_k", [False, True])
@pytest.mark.parametrize("T,C", [(64, 16), (96, 32), (128, 64), (100, 32), (77, 64), (13, 16)])
def test_chunked_backward_equals_token_reverse_mode(per_k, T, C):
    d, do, dhf = problem(per_k, T=T, K=8, seed=T + C)
    n = adjoint(d, do, dhf, C, 0.4)
    c = cb.backward_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], do, dhf, C, 0.4)
    for name in GRADS:
        assert rel(c[name], n[name]) <= 1e-10, name


@pytest.mark.parametrize("per_k", [False, True])
def test_chunked_backward_without_final_gradient(per_k):
    d, do, _ = problem(per_k, T=64, seed=9)
    n = adjoint(d, do, None, 32, 0.4)
    c = cb.backward_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], do, None, 32, 0.4)
    for name in GRADS:
        assert rel(c[name], n[name]) <= 1e-10, name


def test_chunked_stage_invariants():
    d, do, dhf = problem(True, T=64, seed=10)
    r = cb.backward_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], do, dhf, 16, 0.4)
    np.testing.assert_array_equal(r["dh_ckpt"][:, -1], dhf)          # the last chunk sees dh_final
    # dg is the reverse cumsum of dG within each chunk: its chunk-first rows hold the chunk sums
    np.testing.assert_allclose(r["dg"][:, ::16], r["dG"].reshape(2, 4, 16, 2, 6).sum(axis=2), atol=1e-12)


# ---------------------------------------------------------------- grouped value heads

def grouped_problem(per_k, *, B=1, T=9, H=1, G=2, K=3, V=2, seed=60):
    d, do, dhf = problem(per_k, B=B, T=T, H=H * G, K=K, V=V, seed=seed)
    rng = np.random.default_rng(seed)
    d["q"] = rng.standard_normal((B, T, H, K))
    d["k"] = rng.standard_normal((B, T, H, K)) / np.sqrt(K)
    return d, do, dhf


@pytest.mark.parametrize("per_k", [False, True])
def test_grouped_adjoint_matches_finite_differences(per_k):
    # dq and dk of a shared head are the sums over its group: checked against central
    # differences of the grouped forward
    d, do, dhf = grouped_problem(per_k)

    def loss():
        r = oracle.naive_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 4, 0.6, with_ckpt=False)
        return float((r["o"] * do).sum() + (r["h_final"] * dhf).sum())

    got = adjoint(d, do, dhf, 4, 0.6)
    assert got["dq"].shape == d["q"].shape and got["dk"].shape == d["k"].shape
    for name in GRADS:
        x = d[INPUT_OF[name]]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + 1e-6
            lp = loss()
            x[idx] = old - 1e-6
            lm = loss()
            x[idx] = old
            fd[idx] = (lp - lm) / 2e-6
        assert rel(got[name], fd) <= 1e-7, name


@pytest.mark.parametrize("per_k", [False, True])
def test_grouped_chunked_backward_equals_token_reverse_mode(per_k):
    d, do, dhf = grouped_problem(per_k, B=2, T=70, H=2, G=2, K=6, V=5, seed=61)
    n = adjoint(d, do, dhf, 16, 0.4)
    c = cb.backward_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], do, dhf, 16, 0.4)
    for name in GRADS:
        assert rel(c[name], n[name]) <= 1e-10, name
