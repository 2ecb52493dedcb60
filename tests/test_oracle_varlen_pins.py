"""Pins for the packed variable-length oracle (oracle/varlen.py).

A packed batch is n independent problems laid end to end.  The pins check that
reading against things the per-sequence loop does not share: the chunked numpy
oracle on the equivalent batch, a closed form for one-token sequences, the
independence of the sequences (a change in one moves no other), the state an
empty sequence passes through, and, for the backward, central finite
differences of the packed forward.
"""
import numpy as np
import pytest
import torch

from oracle import chunked, varlen
from chunked_gated_delta_prepare_gb300.inputs import make_varlen_inputs


def packed(lengths, per_k, *, H=2, K=6, V=5, HV=None, seed=0, h0_scale=10.0):
    x = make_varlen_inputs(lengths, H, K, V, HV=HV, per_k_gate=per_k, io_dtype=torch.float32, with_h0=True,
                           seed=seed)
    d = {n: t.double().numpy() for n, t in x.tensors().items()}
    d["h0"] = d["h0"] * h0_scale
    return d, x.cu.numpy()


def run(d, cu, C, scale):
    return varlen.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, d["h0"], C, scale)


@pytest.mark.parametrize("per_k", [False, True])
def test_one_sequence_is_the_chunked_problem(per_k):
    d, cu = packed([77], per_k, seed=1)
    o, hf = run(d, cu, 16, 0.5)
    r = chunked.forward_chunked(*(d[n][None] for n in ("q", "k", "v", "g", "beta")), d["h0"], 16, 0.5)
    np.testing.assert_allclose(o, r["o"][0], atol=1e-10)
    np.testing.assert_allclose(hf, r["h_final"], atol=1e-10)


@pytest.mark.parametrize("per_k", [False, True])
def test_equal_lengths_are_the_batch(per_k):
    L, n = 40, 3
    d, cu = packed([L] * n, per_k, seed=2)
    o, hf = run(d, cu, 16, 0.4)
    batch = [d[nm].reshape((n, L) + d[nm].shape[1:]) for nm in ("q", "k", "v", "g", "beta")]
    r = chunked.forward_chunked(*batch, d["h0"], 16, 0.4)
    np.testing.assert_allclose(o, r["o"].reshape(o.shape), atol=1e-10)
    np.testing.assert_allclose(hf, r["h_final"], atol=1e-10)


@pytest.mark.parametrize("per_k", [False, True])
def test_sequences_do_not_see_each_other(per_k):
    lengths = [19, 40, 7]
    d, cu = packed(lengths, per_k, seed=3)
    o, hf = run(d, cu, 16, 0.5)
    # redraw sequence 1's tokens and its initial state
    e, _ = packed(lengths, per_k, seed=99)
    a, b = int(cu[1]), int(cu[2])
    for nm in ("q", "k", "v", "g", "beta"):
        d[nm][a:b] = e[nm][a:b]
    d["h0"][1] = e["h0"][1]
    o2, hf2 = run(d, cu, 16, 0.5)
    assert np.array_equal(o2[:a], o[:a]) and np.array_equal(o2[b:], o[b:])
    assert np.array_equal(hf2[0], hf[0]) and np.array_equal(hf2[2], hf[2])
    assert np.abs(o2[a:b] - o[a:b]).max() > 1e-3 and np.abs(hf2[1] - hf[1]).max() > 1e-3


def test_one_token_sequences_closed_form():
    # a sequence of one token: h = a h0 + beta k (v - a h0^T k)^T with a = e^g, o = scale h^T q
    d, cu = packed([1, 1, 1], False, H=1, K=4, V=3, seed=4)
    scale = 0.7
    o, hf = run(d, cu, 16, scale)
    for s in range(3):
        q, k, v = d["q"][s, 0], d["k"][s, 0], d["v"][s, 0]
        a, beta, h0 = np.exp(d["g"][s, 0]), d["beta"][s, 0], d["h0"][s, 0]
        h = a * h0 + beta * np.outer(k, v - a * h0.T @ k)
        np.testing.assert_allclose(hf[s, 0], h, atol=1e-13)
        np.testing.assert_allclose(o[s, 0], scale * h.T @ q, atol=1e-13)


@pytest.mark.parametrize("per_k", [False, True])
def test_empty_sequence_passes_its_state(per_k):
    d, cu = packed([5, 0, 3, 0], per_k, seed=5)
    o, hf = run(d, cu, 16, 0.5)
    np.testing.assert_array_equal(hf[1], d["h0"][1])
    np.testing.assert_array_equal(hf[3], d["h0"][3])
    o13, hf13 = varlen.forward(*(d[n] for n in ("q", "k", "v", "g", "beta")), np.array([0, 5, 8]),
                               d["h0"][[0, 2]], 16, 0.5)
    np.testing.assert_array_equal(o, o13)
    np.testing.assert_array_equal(hf[[0, 2]], hf13)


@pytest.mark.parametrize("per_k", [False, True])
def test_grouped_heads_are_the_chunked_problem(per_k):
    d, cu = packed([23, 9], per_k, H=1, HV=2, seed=6)
    o, hf = run(d, cu, 8, 0.5)
    for s, (a, b) in enumerate(((0, 23), (23, 32))):
        r = chunked.forward_chunked(*(d[n][None, a:b] for n in ("q", "k", "v", "g", "beta")), d["h0"][s:s + 1], 8,
                                    0.5)
        np.testing.assert_allclose(o[a:b], r["o"][0], atol=1e-10)
        np.testing.assert_allclose(hf[s], r["h_final"][0], atol=1e-10)


@pytest.mark.parametrize("per_k", [False, True])
def test_backward_matches_finite_differences(per_k):
    lengths = [3, 0, 2]
    d, cu = packed(lengths, per_k, H=1, K=3, V=2, seed=7, h0_scale=30.0)
    scale = 0.7
    rng = np.random.default_rng(8)
    do = rng.standard_normal(d["v"].shape)
    dhf = rng.standard_normal(d["h0"].shape)

    def loss():
        o, hf = run(d, cu, 2, scale)
        return float((o * do).sum() + (hf * dhf).sum())

    got = varlen.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, d["h0"], do, dhf, 2, scale)
    for name, inp in (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dg", "g"), ("dbeta", "beta"), ("dh0", "h0")):
        x = d[inp]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + 1e-6
            lp = loss()
            x[idx] = old - 1e-6
            lm = loss()
            x[idx] = old
            fd[idx] = (lp - lm) / 2e-6
        np.testing.assert_allclose(got[name], fd, atol=1e-6, rtol=1e-6, err_msg=name)


def test_cu_must_start_at_zero_and_not_decrease():
    d, _ = packed([4, 4], False, seed=9)
    for bad in ([1, 4, 8], [0, 5, 4]):
        with pytest.raises(ValueError):
            run(d, np.array(bad), 16, 0.5)


@pytest.mark.parametrize("per_k", [False, True])
def test_backward_equal_lengths_are_the_chunked_batch(per_k):
    # the packed reverse mode (the C adjoint per sequence) against the chunked numpy backward on the
    # reshaped batch, a formulation it shares nothing with
    from oracle import chunked_backward
    L, n = 40, 3
    d, cu = packed([L] * n, per_k, K=6, V=5, seed=10)
    rng = np.random.default_rng(11)
    do = rng.standard_normal(d["v"].shape)
    dhf = rng.standard_normal(d["h0"].shape)
    got = varlen.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, d["h0"], do, dhf, 16, 0.4)
    batch = {nm: d[nm].reshape((n, L) + d[nm].shape[1:]) for nm in ("q", "k", "v", "g", "beta")}
    ref = chunked_backward.backward_chunked(batch["q"], batch["k"], batch["v"], batch["g"], batch["beta"], d["h0"],
                                            do.reshape((n, L) + do.shape[1:]), dhf, 16, 0.4)
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        np.testing.assert_allclose(got[name], ref[name].reshape(got[name].shape), atol=1e-9, err_msg=name)
    np.testing.assert_allclose(got["dh0"], ref["dh0"], atol=1e-9)
