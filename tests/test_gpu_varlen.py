"""Packed variable-length sequences on the GPU: gdr_varlen_forward and
gdr_varlen_backward (through the C ABI) against the float64 per-sequence oracle
(oracle/varlen.py) on the same rounded inputs.

The bars are those of the batched calls: forward o max-abs 2e-2 and h_final
relative Frobenius 1e-2 for bf16 and fp16 io, 1e-4 for fp32; backward max |x - ref| /
max |ref| per gradient 2e-2 for bf16 and 1e-4 for fp32.  Each padded row runs
the batched kernels, so the same rounding steps apply.  Output buffers start as
NaN, so a packed row the call fails to write fails the comparison.
"""
import numpy as np
import pytest
import torch

from oracle import varlen
from chunked_gated_delta_prepare_gb300 import gdr
from chunked_gated_delta_prepare_gb300.inputs import make_varlen_inputs
from gpu_helpers import H_TOL, O_TOL, dev, io_name, max_abs, rel_frob, scaled_err

pytestmark = pytest.mark.gpu

BWD_TOL = {"bf16": 2e-2, "f16": 2e-2, "f32": 1e-4}
# empty, one-token, partial-chunk, exact-chunk and several-chunk sequences side by side
MIXED = [100, 0, 1, 64, 200, 63, 65, 31]
PATHS = [("simt", torch.float32, False), ("simt", torch.float32, True), ("tensor", torch.bfloat16, False),
         ("tensor", torch.bfloat16, True), ("fused", torch.bfloat16, False), ("auto", torch.bfloat16, False),
         ("auto", torch.bfloat16, True), ("simt", torch.float16, False), ("tensor", torch.float16, False),
         ("tensor", torch.float16, True), ("fused", torch.float16, False), ("auto", torch.float16, True)]
SCALE = 0.09


def inputs(lengths, per_k, dtype, *, H=2, HV=None, K=64, V=64, seed=0):
    return make_varlen_inputs(lengths, H, K, V, HV=HV, per_k_gate=per_k, io_dtype=dtype, with_h0=True, seed=seed)


def gpu_forward(x, C, variant, *, device_cu=False, max_len=None):
    q, k, v, g, beta, h0 = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.h0))
    cu = x.cu.to("cuda") if device_cu else x.cu
    p = gdr.varlen_problem(q, v, g, x.cu, max_len, C, SCALE, variant, 0)
    n, K, HV, V = int(p.B), q.shape[-1], v.shape[-2], v.shape[-1]
    o = torch.full(v.shape, float("nan"), device="cuda", dtype=v.dtype)
    hf = torch.full((n, HV, K, V), float("nan"), device="cuda")
    nbytes = gdr.gdr_varlen_forward_workspace_bytes(p)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    gdr.gdr_varlen_forward(p, x.cu, cu if device_cu else None, int(x.cu[-1]), q, k, v, g, beta, h0, o, hf, ws,
                           nbytes)
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    return o, hf, gdr.gdr_last_variant()


def reference(x, C):
    d = {n: None if t is None else t.double().numpy() for n, t in x.tensors().items()}
    return varlen.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], x.cu.numpy(), d["h0"], C, SCALE)


@pytest.mark.parametrize("variant,dtype,per_k", PATHS)
@pytest.mark.parametrize("C", [32, 64])
def test_varlen_forward_mixed_lengths(variant, dtype, per_k, C):
    x = inputs(MIXED, per_k, dtype, K=64 if C == 32 else 128, V=128 if C == 32 else 64, seed=C)
    o, hf, var = gpu_forward(x, C, variant)
    o_ref, hf_ref = reference(x, C)
    io = io_name(dtype)
    assert max_abs(o, o_ref) <= O_TOL[io], (var, max_abs(o, o_ref))
    assert rel_frob(hf, hf_ref) <= H_TOL[io], (var, rel_frob(hf, hf_ref))
    if variant != "auto":
        assert var == variant


@pytest.mark.parametrize("per_k", [False, True])
def test_varlen_grouped_heads_and_device_cu(per_k):
    x = inputs([70, 128, 5, 0, 191], per_k, torch.bfloat16, H=1, HV=3, seed=5)
    o, hf, _ = gpu_forward(x, 64, "auto")
    o2, hf2, _ = gpu_forward(x, 64, "auto", device_cu=True)
    assert torch.equal(o, o2) and torch.equal(hf, hf2)
    o_ref, hf_ref = reference(x, 64)
    assert max_abs(o, o_ref) <= O_TOL["bf16"] and rel_frob(hf, hf_ref) <= H_TOL["bf16"]


def test_varlen_longer_rows_change_nothing():
    # rows longer than the longest sequence only add zero tokens
    x = inputs(MIXED, False, torch.bfloat16, K=128, V=128, seed=7)
    o, hf, _ = gpu_forward(x, 64, "tensor")
    o2, hf2, _ = gpu_forward(x, 64, "tensor", max_len=448)
    o_ref, hf_ref = reference(x, 64)
    for a, b in ((o, hf), (o2, hf2)):
        assert max_abs(a, o_ref) <= O_TOL["bf16"] and rel_frob(b, hf_ref) <= H_TOL["bf16"]


def test_varlen_all_sequences_empty():
    x = inputs([0, 0, 0], False, torch.bfloat16, K=128, V=128, seed=8)
    o, hf, _ = gpu_forward(x, 64, "auto")
    assert o.numel() == 0
    np.testing.assert_allclose(hf.cpu().numpy(), x.h0.numpy(), rtol=0, atol=1e-7)


def test_varlen_rejects_bad_cu_before_launching():
    x = inputs([10, 20], False, torch.bfloat16, K=128, V=128, seed=9)
    q, k, v, g, beta = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta))
    p = gdr.make_problem(2, 15, 1, 128, 128, 64, torch.bfloat16, False)      # rows shorter than sequence 1
    nbytes = gdr.gdr_varlen_forward_workspace_bytes(p)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    o = torch.empty_like(v)
    with pytest.raises(gdr.GdrError) as e:
        gdr.gdr_varlen_forward(p, x.cu, None, 30, q, k, v, g, beta, None, o, None, ws, nbytes)
    assert e.value.status == 9


def test_convenience_forward_varlen():
    x = inputs(MIXED, True, torch.bfloat16, H=2, K=128, V=128, seed=10)
    q, k, v, g, beta, h0 = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.h0))
    o, hf = gdr.forward_varlen(q, k, v, g, beta, x.cu.tolist(), h0, chunk=64, scale=SCALE)
    o_ref, hf_ref = reference(x, 64)
    assert max_abs(o, o_ref) <= O_TOL["bf16"] and rel_frob(hf, hf_ref) <= H_TOL["bf16"]


# ---------------------------------------------------------------- backward

def upstream(x, seed):
    gen = torch.Generator().manual_seed(seed)
    n = x.cu.numel() - 1
    HV, K, V = x.v.shape[-2], x.k.shape[-1], x.v.shape[-1]
    return torch.randn(x.v.shape, generator=gen).to(x.v.dtype), torch.randn(n, HV, K, V, generator=gen)


# the backward: no fused variant, and fp16 on the CUDA-core kernels only (TENSOR refuses it)
BWD_PATHS = [p for p in PATHS if p[0] != "fused" and not (p[1] == torch.float16 and p[0] == "tensor")]


@pytest.mark.parametrize("variant,dtype,per_k", BWD_PATHS)
@pytest.mark.parametrize("C", [32, 64])
def test_varlen_backward_mixed_lengths(variant, dtype, per_k, C):
    x = inputs(MIXED, per_k, dtype, K=64 if C == 32 else 128, V=128 if C == 32 else 64, seed=20 + C)
    do, dhf = upstream(x, 3)
    q, k, v, g, beta, h0 = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.h0))
    dq, dk, dv, dg, dbeta, dh0 = gdr.backward_varlen(q, k, v, g, beta, x.cu, h0, dev(do), dev(dhf), chunk=C,
                                                     scale=SCALE, variant=variant)
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    d = {n_: t.double().numpy() for n_, t in x.tensors().items()}
    ref = varlen.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], x.cu.numpy(), d["h0"], do.double().numpy(),
                          dhf.double().numpy(), C, SCALE)
    tol = BWD_TOL[io_name(dtype)]
    for name, got in zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), (dq, dk, dv, dg, dbeta, dh0)):
        assert scaled_err(got, ref[name]) <= tol, (name, scaled_err(got, ref[name]))


# ---------------------------------------------------------------- a long packed batch

def test_varlen_long_mixed_batch_sampled_heads():
    # 32 heads of 128 x 128 over 32k packed tokens in eleven sequences (one empty, ragged tails); the
    # oracle recomputes two of the heads
    lengths = [8192, 4096, 4133, 1, 6000, 0, 2048, 3000, 777, 2911, 1610]
    H, K, V, C = 32, 128, 128, 64
    x = inputs(lengths, False, torch.bfloat16, H=H, K=K, V=V, seed=11)
    o, hf, _ = gpu_forward(x, C, "auto")
    heads = [3, 30]
    sub = make_varlen_inputs(lengths, H, K, V, io_dtype=torch.bfloat16, with_h0=True, seed=11)
    for name in ("q", "k", "v", "g", "beta"):
        setattr(sub, name, getattr(sub, name)[:, heads].contiguous())
    sub.h0 = sub.h0[:, heads].contiguous()
    o_ref, hf_ref = reference(sub, C)
    assert max_abs(o[:, heads], o_ref) <= O_TOL["bf16"]
    assert rel_frob(hf[:, heads], hf_ref) <= H_TOL["bf16"]


def test_varlen_backward_long_mixed_batch_sampled_heads():
    # 32 heads of 128 x 128 over 8k packed tokens in six sequences; the oracle recomputes two heads
    lengths = [2048, 1, 0, 3000, 777, 2366]
    H, K, V, C = 32, 128, 128, 64
    x = inputs(lengths, False, torch.bfloat16, H=H, K=K, V=V, seed=12)
    do, dhf = upstream(x, 4)
    q, k, v, g, beta, h0 = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.h0))
    got = gdr.backward_varlen(q, k, v, g, beta, x.cu, h0, dev(do), dev(dhf), chunk=C, scale=SCALE)
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    assert gdr.gdr_last_variant() == "tensor"
    heads = [5, 27]
    d = {n_: t[:, heads].double().numpy() for n_, t in x.tensors().items()}
    ref = varlen.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], x.cu.numpy(), d["h0"],
                          do[:, heads].double().numpy(), dhf[:, heads].double().numpy(), C, SCALE)
    for name, t in zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), got):
        assert scaled_err(t[:, heads], ref[name]) <= BWD_TOL["bf16"], (name, scaled_err(t[:, heads], ref[name]))


@pytest.mark.parametrize("per_k", [False, True])
def test_varlen_many_short_sequences(per_k):
    # 2500 sequences of 0 to 70 tokens: the chunk map's prefix sum runs over several 1024-sequence tiles
    lengths = np.random.default_rng(13).integers(0, 71, size=2500).tolist()
    x = inputs(lengths, per_k, torch.bfloat16, H=2, K=64, V=64, seed=13)
    o, hf, var = gpu_forward(x, 64, "auto")
    assert var == ("tensor" if per_k else "fused")
    o_ref, hf_ref = reference(x, 64)
    assert max_abs(o, o_ref) <= O_TOL["bf16"] and rel_frob(hf, hf_ref) <= H_TOL["bf16"]
    do, dhf = upstream(x, 5)
    q, k, v, g, beta, h0 = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.h0))
    got = gdr.backward_varlen(q, k, v, g, beta, x.cu, h0, dev(do), dev(dhf), chunk=64, scale=SCALE)
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    d = {n_: t.double().numpy() for n_, t in x.tensors().items()}
    ref = varlen.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], x.cu.numpy(), d["h0"], do.double().numpy(),
                          dhf.double().numpy(), 64, SCALE)
    for name, t in zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), got):
        assert scaled_err(t, ref[name]) <= BWD_TOL["bf16"], (name, scaled_err(t, ref[name]))


@pytest.mark.parametrize("variant,C", [("fused", 64), ("fused", 32), ("tensor", 64)])
def test_varlen_sequences_are_isolated_from_nonfinite_neighbours(variant, C):
    # the fused path at C = 64 reads the packed tensors in place, so a sequence's last chunk sees the next
    # sequence's tokens in its tail rows until they are zeroed: an inf or a NaN there must not leak
    lengths = [100, 37, 70]
    x = inputs(lengths, False, torch.bfloat16, H=2, K=128, V=128, seed=14)
    o, hf, _ = gpu_forward(x, C, variant)
    a, b = int(x.cu[1]), int(x.cu[2])
    x.k[a:b] = float("nan")
    x.q[a:b] = float("inf")
    x.v[a:b] = float("nan")
    o2, hf2, _ = gpu_forward(x, C, variant)
    assert torch.equal(o2[:a], o[:a]) and torch.equal(o2[b:], o[b:])
    assert torch.equal(hf2[0], hf[0]) and torch.equal(hf2[2], hf[2])
