"""Backward parity on the GPU: gdr_backward and its four stage entry points
(through the C ABI) against the float64 backward oracles on the same rounded inputs.

Tolerances (max |x - ref| / max |ref| per gradient tensor).
- fp32 io: 1e-4. Every product and sum is fp32, and sums run over at most a few
  hundred terms per stage; that is the forward's fp32 class.
- bf16 io: 2e-2. The re-scan keeps w, u, v' and the checkpoints in bf16, each
  a 2^-9 relative rounding, and each gradient term is a product of up to three
  such factors plus a bf16 store: about 4 x 2^-9, the forward's bf16 o bar.
Per-stage tests feed each stage the oracle's own intermediates, rounded as the
library stores them, so only that stage's arithmetic is compared.  Their bars
are the per-stage classes of the forward: 1e-5 for fp32 and 1e-2 for bf16.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from oracle import chunked, chunked_backward as cb
from chunked_gated_delta_prepare_gb300 import gdr, workloads
from chunked_gated_delta_prepare_gb300.inputs import GdrInputs, make_inputs, make_workload_inputs
from gpu_helpers import STAGE_TOL, all_pairs, dev, gather_heads, grouped_inputs, io_name, sample_heads, scaled_err

pytestmark = pytest.mark.gpu

BWD_TOL = {"bf16": 2e-2, "f16": 2e-2, "f32": 1e-4}
GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dh0")
# (B, T, H, K, V, C): several chunks, both chunk sizes, K != V, and partial last chunks
SHAPES = [(2, 256, 3, 64, 64, 64), (1, 192, 2, 128, 128, 64), (2, 128, 3, 64, 128, 32),
          (1, 160, 1, 128, 64, 32), (2, 100, 2, 64, 64, 64), (1, 77, 2, 128, 128, 32), (1, 20, 1, 64, 64, 64)]
VARIANTS = {"simt": (torch.float32, torch.bfloat16), "tensor": (torch.bfloat16,)}


def upstream(x, seed):
    """do (io dtype) and dh_final (fp32) for the inputs x, seeded."""
    gen = torch.Generator().manual_seed(seed)
    B, T, H = x.v.shape[:3]
    K, V = x.k.shape[-1], x.v.shape[-1]
    do = torch.randn(B, T, H, V, generator=gen).to(x.q.dtype)
    dhf = torch.randn(B, H, K, V, generator=gen)
    return do, dhf


def gpu_backward(x, do, dhf, C, variant, scale=None, want_dh0=True, segments=0):
    q, k, v, g, beta, h0, d_o = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.h0, do))
    p = gdr.problem_for(q, v, g, C, scale, variant, segments)
    B, T, _, K = q.shape
    H, V = v.shape[2], v.shape[-1]            # value heads
    nan = float("nan")
    outs = dict(dq=torch.full_like(q, nan), dk=torch.full_like(k, nan), dv=torch.full_like(v, nan),
                dg=torch.full_like(g, nan), dbeta=torch.full_like(beta, nan),
                dh0=torch.full((B, H, K, V), nan, device="cuda") if want_dh0 else None)
    nbytes = gdr.gdr_backward_workspace_bytes(p)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    gdr.gdr_backward(p, q, k, v, g, beta, h0, d_o, dev(dhf), outs["dq"], outs["dk"], outs["dv"], outs["dg"],
                     outs["dbeta"], outs["dh0"], ws, nbytes)
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    return outs, gdr.gdr_last_variant()


def reference(x, do, dhf, C, scale):
    return oracle.naive_backward(x.q, x.k, x.v, x.g, x.beta, x.h0, do, dhf, C, scale)


def cases():
    for shape, per_k, (variant, dts) in itertools.product(SHAPES, (False, True), VARIANTS.items()):
        for dt in dts:
            yield pytest.param(shape, per_k, variant, dt,
                               id=f"{'x'.join(map(str, shape))}-{'kda' if per_k else 'gdn'}-{variant}-{io_name(dt)}")


@pytest.mark.parametrize("shape,per_k,variant,dtype", list(cases()))
def test_backward_against_token_reverse_mode(shape, per_k, variant, dtype):
    B, T, H, K, V, C = shape
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=dtype, with_h0=True, seed=40)
    do, dhf = upstream(x, 41)
    scale = 1.0 / np.sqrt(K)
    got, ran = gpu_backward(x, do, dhf, C, variant)
    assert ran == variant
    ref = reference(x, do, dhf, C, scale)
    for name in GRADS:
        err = scaled_err(got[name], ref[name])
        assert np.isfinite(err) and err <= BWD_TOL[io_name(dtype)], f"{name}: {err:.3e}"


@pytest.mark.parametrize("per_k", [False, True])
def test_backward_without_final_gradient_or_dh0(per_k):
    x = make_inputs(1, 128, 2, 64, 64, per_k_gate=per_k, io_dtype=torch.float32, with_h0=True, seed=42)
    do, _ = upstream(x, 43)
    got, _ = gpu_backward(x, do, None, 32, "simt", want_dh0=False)
    ref = reference(x, do, None, 32, 1 / 8.0)
    for name in GRADS[:-1]:
        assert scaled_err(got[name], ref[name]) <= BWD_TOL["f32"], name


def _edge(kind, per_k, dtype):
    x = make_inputs(1, 96, 2, 64, 64, per_k_gate=per_k, io_dtype=dtype, with_h0=True, seed=44)
    g, beta = x.g.clone(), x.beta.clone()
    if kind == "beta_zero":
        beta.zero_()
    elif kind == "no_decay":
        g.zero_()
    elif kind == "strong_decay":
        g.fill_(-20.0)
    elif kind == "single_token":
        return GdrInputs(q=x.q[:, :1], k=x.k[:, :1], v=x.v[:, :1], g=x.g[:, :1], beta=x.beta[:, :1], h0=x.h0 * 20)
    return GdrInputs(q=x.q, k=x.k, v=x.v, g=g, beta=beta, h0=x.h0 * 20)


@pytest.mark.parametrize("kind", ["beta_zero", "no_decay", "strong_decay", "single_token"])
@pytest.mark.parametrize("variant,dtype,per_k", [(v, d, pk) for v, ds in VARIANTS.items() for d in ds
                                                  for pk in (False, True)])
def test_backward_edge_cases(kind, variant, dtype, per_k):
    x = _edge(kind, per_k, dtype)
    do, dhf = upstream(x, 45)
    got, _ = gpu_backward(x, do, dhf, 32, variant)
    ref = reference(x, do, dhf, 32, 1 / 8.0)
    for name in GRADS:
        if np.abs(ref[name]).max() == 0.0:
            assert float(got[name].abs().max()) == 0.0, name
            continue
        assert scaled_err(got[name], ref[name]) <= BWD_TOL[io_name(dtype)], name


def test_backward_refuses_fused_and_small_workspace():
    x = make_inputs(1, 64, 1, 64, 64, io_dtype=torch.bfloat16, seed=46)
    p = gdr.problem_for(x.q, x.v, x.g, 64, variant="fused")
    assert gdr.gdr_backward_workspace_bytes(p) == 0
    t = torch.zeros(64, 1, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(gdr.GdrError) as e:
        gdr.gdr_backward(p, t, t, t, t, t, None, t, None, t, t, t, t, t, None, t, 1 << 30)
    assert e.value.status == 8
    p = gdr.problem_for(x.q, x.v, x.g, 64, variant="tensor")
    need = gdr.gdr_backward_workspace_bytes(p)
    ws = torch.empty(need, device="cuda", dtype=torch.uint8)
    with pytest.raises(gdr.GdrError) as e:
        gdr.gdr_backward(p, t, t, t, t, t, None, t, None, t, t, t, t, t, None, ws, need - 1)
    assert e.value.status == 5


def test_convenience_backward():
    x = make_inputs(2, 128, 2, 64, 64, io_dtype=torch.bfloat16, with_h0=True, seed=47)
    do, dhf = upstream(x, 48)
    args = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.h0, do, dhf))
    dq, dk, dv, dg, dbeta, dh0 = gdr.backward(*args, chunk=64)
    ref = reference(x, do, dhf, 64, 1 / 8.0)
    for name, t in zip(GRADS, (dq, dk, dv, dg, dbeta, dh0)):
        assert scaled_err(t, ref[name]) <= BWD_TOL["bf16"], name


# The named workloads at full size through gdr_backward (variant AUTO, as the
# benchmark runs it); heads are sampled where the oracle would be slow, and every
# token of a sampled head is checked.
BWD_SAMPLES = {workloads.KDA_BF16_T8K.name: [(0, 0), (1, 15)], workloads.GDN_BF16_T32K.name: [(0, 0), (0, 31)]}


@pytest.mark.parametrize("wl", workloads.ALL, ids=lambda w: w.name)
def test_backward_workload_full_size(wl):
    x = make_workload_inputs(wl)
    do, dhf = upstream(x, 60)
    got, ran = gpu_backward(x, do, dhf, wl.chunk, "auto")
    pairs = BWD_SAMPLES.get(wl.name) or all_pairs(wl.B, wl.H)
    s = sample_heads(x, pairs)
    d_o = torch.stack([do[b, :, h] for b, h in pairs]).unsqueeze(2)
    dh = torch.stack([dhf[b, h] for b, h in pairs]).unsqueeze(1)
    ref = oracle.naive_backward(s["q"], s["k"], s["v"], s["g"], s["beta"], s["h0"], d_o, dh, wl.chunk,
                                1.0 / np.sqrt(wl.K))
    errs = {}
    for name in GRADS:
        errs[name] = scaled_err(gather_heads(got[name], pairs, state=name == "dh0"), ref[name])
        assert np.isfinite(errs[name]) and errs[name] <= BWD_TOL[wl.io], f"{name}: {errs[name]:.3e}"
    print(f"{wl.name}: variant={ran} " + " ".join(f"{n} {e:.1e}" for n, e in errs.items()))


# ---------------------------------------------------------------- stages

STAGE_SHAPES = [(2, 128, 3, 64, 64, 64), (1, 192, 2, 128, 128, 64), (2, 96, 1, 64, 128, 32), (1, 77, 2, 128, 64, 32)]


def rounded(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype)


def stage_cases():
    for shape, per_k, dt in itertools.product(STAGE_SHAPES, (False, True), (torch.float32, torch.bfloat16)):
        yield pytest.param(shape, per_k, dt, id=f"{'x'.join(map(str, shape))}-{'kda' if per_k else 'gdn'}-{io_name(dt)}")


def _stage_setup(shape, per_k, dtype, seed):
    B, T, H, K, V, C = shape
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=dtype, with_h0=True, seed=seed)
    do, dhf = upstream(x, seed + 1)
    h0 = x.h0 * 20
    full = cb.backward_chunked(x.q, x.k, x.v, x.g, x.beta, h0, do, dhf, C, 0.125)
    p = gdr.problem_for(x.q, x.v, x.g, C, scale=0.125, variant="simt")
    return x, do, dhf, full, p


@pytest.mark.parametrize("shape,per_k,dtype", list(stage_cases()))
def test_stage_dv_local(shape, per_k, dtype):
    x, do, _, full, p = _stage_setup(shape, per_k, dtype, 50)
    G_r = rounded(full["G"], torch.float32)
    ref = cb.dv_local(x.q, x.k, G_r, do, shape[-1], 0.125)
    out = torch.full(x.v.shape, float("nan"), device="cuda")
    gdr.gdr_bwd_dv_local(p, dev(x.q), dev(x.k), dev(G_r), dev(do), out)
    torch.cuda.synchronize()
    assert scaled_err(out, ref) <= STAGE_TOL[io_name(dtype)]


@pytest.mark.parametrize("shape,per_k,dtype", list(stage_cases()))
def test_stage_scan_dh(shape, per_k, dtype):
    x, do, dhf, full, p = _stage_setup(shape, per_k, dtype, 52)
    B, T, H, K, V, C = shape
    G_r, w_r = rounded(full["G"], torch.float32), rounded(full["w"], dtype)
    dl = rounded(full["dv_local"], torch.float32)
    ref = cb.scan_dh(x.q, x.k, w_r, G_r, do, dl, dhf, C, 0.125)
    NT = -(-T // C)
    dh_ckpt = torch.full((B, NT, H, K, V), float("nan"), device="cuda")
    dv_new = torch.full((B, T, H, V), float("nan"), device="cuda")
    dh0 = torch.full((B, H, K, V), float("nan"), device="cuda")
    gdr.gdr_bwd_scan_dh(p, dev(x.q), dev(x.k), dev(w_r), dev(G_r), dev(do), dev(dl), dev(dhf), dh_ckpt, dv_new, dh0)
    torch.cuda.synchronize()
    tol = STAGE_TOL[io_name(dtype)]
    assert scaled_err(dh_ckpt, ref["dh_ckpt"]) <= tol
    assert scaled_err(dv_new, ref["dv_new"]) <= tol
    assert scaled_err(dh0, ref["dh0"]) <= tol


@pytest.mark.parametrize("shape,per_k,dtype", list(stage_cases()))
def test_stage_dqkwg(shape, per_k, dtype):
    x, do, _, full, p = _stage_setup(shape, per_k, dtype, 54)
    B, T, H, K, V, C = shape
    G_r, w_r = rounded(full["G"], torch.float32), rounded(full["w"], dtype)
    vn_r, hc_r = rounded(full["v_new"], dtype), rounded(full["h_ckpt"], dtype)
    dhc, dvn = rounded(full["dh_ckpt"], torch.float32), rounded(full["dv_new"], torch.float32)
    ref = cb.dqkwg(x.q, x.k, vn_r, w_r, G_r, hc_r, dhc, do, dvn, C, 0.125)
    nan = float("nan")
    dq = torch.full(x.q.shape, nan, device="cuda", dtype=dtype)
    dk_part = torch.full(x.k.shape, nan, device="cuda")
    dw = torch.full(x.k.shape, nan, device="cuda")
    dG = torch.full(x.g.shape, nan, device="cuda")
    gdr.gdr_bwd_dqkwg(p, dev(x.q), dev(x.k), dev(vn_r), dev(G_r), dev(hc_r), dev(dhc), dev(do), dev(dvn),
                      dq, dk_part, dw, dG)
    torch.cuda.synchronize()
    tol = STAGE_TOL[io_name(dtype)]
    assert scaled_err(dq, ref["dq"]) <= tol
    assert scaled_err(dk_part, ref["dk"]) <= tol
    assert scaled_err(dw, ref["dw"]) <= tol
    assert scaled_err(dG, ref["dG"] if per_k else ref["dG"].sum(-1)) <= tol


@pytest.mark.parametrize("shape,per_k,dtype", list(stage_cases()))
def test_stage_wy(shape, per_k, dtype):
    x, do, _, full, p = _stage_setup(shape, per_k, dtype, 56)
    B, T, H, K, V, C = shape
    G_r = rounded(full["G"], torch.float32)
    dw, du = rounded(full["dw"], torch.float32), rounded(full["dv_new"], torch.float32)
    a = cb.dqkwg(x.q, x.k, full["v_new"], full["w"], full["G"], full["h_ckpt"], full["dh_ckpt"], do,
                 full["dv_new"], C, 0.125)
    dk_part = rounded(a["dk"], torch.float32)
    dG_part = rounded(a["dG"] if per_k else a["dG"].sum(-1), torch.float32)
    y = cb.wy_backward(x.k, x.v, x.beta, G_r, dw, du, C)
    # the gate gradient before the cumsum: per key dim, or (scalar gate) summed over it once
    dG_ref = dG_part.double().numpy() + (y["dG"] if per_k else y["dG"].sum(-1))
    if not per_k:
        dG_ref = dG_ref[..., None]
    nan = float("nan")
    dk = torch.full(x.k.shape, nan, device="cuda", dtype=dtype)
    dv = torch.full(x.v.shape, nan, device="cuda", dtype=dtype)
    dbeta = torch.full(x.beta.shape, nan, device="cuda", dtype=dtype)
    dg = torch.full(x.g.shape, nan, device="cuda")
    gdr.gdr_bwd_wy(p, dev(x.k), dev(x.v), dev(x.beta), dev(G_r), dev(dw), dev(du), dev(dk_part), dev(dG_part),
                   dk, dv, dbeta, dg)
    torch.cuda.synchronize()
    tol = STAGE_TOL[io_name(dtype)]
    assert scaled_err(dk, dk_part.double().numpy() + y["dk"]) <= tol
    assert scaled_err(dv, y["dv"]) <= tol
    assert scaled_err(dbeta, y["dbeta"]) <= tol
    assert scaled_err(dg, cb.reverse_cumsum(dG_ref, C, per_k)) <= tol


# ---------------------------------------------------------------- tensor-core stages (bf16, scalar gate, C = 64)

FAST_SHAPES = [(2, 128, 3, 64, 64, 64), (1, 192, 2, 128, 128, 64), (2, 100, 2, 128, 64, 64), (1, 256, 1, 64, 128, 64)]


def _fast_setup(shape, seed, per_k=False, strong_head=None):
    B, T, H, K, V, C = shape
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=torch.bfloat16, with_h0=True, seed=seed)
    if strong_head is not None:   # one head's gate 100 times stronger: its chunks span far more than e^40
        g = x.g.clone()
        g[:, :, strong_head] *= 100.0
        x = GdrInputs(q=x.q, k=x.k, v=x.v, g=g, beta=x.beta, h0=x.h0)
    do, dhf = upstream(x, seed + 1)
    full = cb.backward_chunked(x.q, x.k, x.v, x.g, x.beta, x.h0 * 20, do, dhf, C, 0.125)
    p = gdr.problem_for(x.q, x.v, x.g, C, scale=0.125, variant="tensor")
    return x, do, dhf, full, p


@pytest.mark.parametrize("shape", FAST_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_tensor_stage_prepare_with_inverse(shape):
    x, _, _, full, p = _fast_setup(shape, 70)
    B, T, H, K, V, C = shape
    NT = -(-T // C)
    q, k, v, g, beta = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta))
    nan = float("nan")
    w, u, g_cum = torch.full_like(k, nan), torch.full_like(v, nan), torch.full_like(g, nan)
    P = torch.full((B, NT, H, C, C), nan, device="cuda", dtype=torch.bfloat16)
    tinv = torch.full((B, NT, H, C, C), nan, device="cuda", dtype=torch.bfloat16)
    gdr.gdr_bwd_prepare(p, q, k, v, g, beta, w, u, g_cum, P, tinv)
    torch.cuda.synchronize()
    assert gdr.gdr_last_variant() == "tensor"
    A = chunked.gated_A(x.k, x.beta, full["G"], C)
    assert scaled_err(tinv, chunked.forward_substitution_inverse(A)) <= STAGE_TOL["bf16"]
    assert scaled_err(P, chunked.gated_causal_scores(x.q, x.k, full["G"], C)) <= STAGE_TOL["bf16"]
    assert scaled_err(w, full["w"]) <= STAGE_TOL["bf16"] and scaled_err(u, full["u"]) <= STAGE_TOL["bf16"]


@pytest.mark.parametrize("shape", FAST_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("with_dhf", [False, True])
def test_tensor_stage_reverse_scan(shape, with_dhf):
    x, do, dhf, full, p = _fast_setup(shape, 72)
    B, T, H, K, V, C = shape
    dhf = dhf if with_dhf else None
    G_r, w_r = rounded(full["G"], torch.float32), rounded(full["w"], torch.bfloat16)
    P_r = rounded(chunked.gated_causal_scores(x.q, x.k, G_r, C), torch.bfloat16)
    dl = cb.dv_local(x.q, x.k, G_r, do, C, 0.125)
    ref = cb.scan_dh(x.q, x.k, w_r, G_r, do, dl, dhf, C, 0.125)
    NT = -(-T // C)
    nan = float("nan")
    dh_ckpt = torch.full((B, NT, H, K, V), nan, device="cuda", dtype=torch.bfloat16)
    dv_new = torch.full((B, T, H, V), nan, device="cuda", dtype=torch.bfloat16)
    dh0 = torch.full((B, H, K, V), nan, device="cuda")
    gdr.gdr_bwd_scan_dh_p(p, dev(x.q), dev(x.k), dev(w_r), dev(G_r), dev(P_r), dev(do), dev(dhf), dh_ckpt, dv_new, dh0)
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    tol = STAGE_TOL["bf16"]
    assert scaled_err(dh_ckpt, ref["dh_ckpt"]) <= tol
    assert scaled_err(dv_new, ref["dv_new"]) <= tol
    assert scaled_err(dh0, ref["dh0"]) <= tol


@pytest.mark.parametrize("shape", FAST_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_tensor_stage_wy_dqkg(shape):
    _wy_dqkg_case(shape)


def _wy_dqkg_case(shape, per_k=False, strong_head=None):
    x, do, _, full, p = _fast_setup(shape, 74, per_k, strong_head)
    B, T, H, K, V, C = shape
    NT = -(-T // C)
    bf = torch.bfloat16
    G_r = rounded(full["G"], torch.float32)
    w_r, u_r, vn_r, hc_r = (rounded(full[n], bf) for n in ("w", "u", "v_new", "h_ckpt"))
    dvn_r, dhc_r = rounded(full["dv_new"], bf), rounded(full["dh_ckpt"], bf)
    A = chunked.gated_A(x.k, x.beta, G_r, C)
    tinv_r = rounded(chunked.forward_substitution_inverse(A), bf)
    a = cb.dqkwg(x.q, x.k, vn_r, w_r, G_r, hc_r, dhc_r, do, dvn_r, C, 0.125)
    y = cb.wy_backward(x.k, x.v, x.beta, G_r, a["dw"], dvn_r, C)
    nan = float("nan")
    dq, dk, dv = torch.full(x.q.shape, nan, device="cuda", dtype=bf), torch.full(x.k.shape, nan, device="cuda",
                                                                                   dtype=bf), \
        torch.full(x.v.shape, nan, device="cuda", dtype=bf)
    dbeta, dg = torch.full(x.beta.shape, nan, device="cuda", dtype=bf), torch.full(x.g.shape, nan, device="cuda")
    flags = torch.full((B, NT, H), -1, device="cuda", dtype=torch.int32) if per_k else None
    args = [dev(x.q), dev(x.k), dev(x.v), dev(x.beta), dev(G_r), dev(w_r), dev(u_r), dev(tinv_r), dev(vn_r),
            dev(hc_r), dev(do), dev(dvn_r), dev(dhc_r)]
    gdr.gdr_bwd_wy_dqkg(p, *args, dq, dk, dv, dbeta, dg, flags)
    if per_k:
        torch.cuda.synchronize()
        f = flags.cpu()
        assert set(f.unique().tolist()) <= {0, 1}
        if strong_head is None:
            assert int(f.sum()) == 0
        else:   # the strong head's chunks, and only they, go to the CUDA-core stages
            assert int(f[:, :, strong_head].sum()) > 0 and int(f.sum()) == int(f[:, :, strong_head].sum())
        # the flagged chunks, exactly in fp32 (the entry points read bf16 intermediates, variant tensor)
        dk_part, dw = torch.empty(x.k.shape, device="cuda"), torch.empty(x.k.shape, device="cuda")
        dG_part = torch.empty(x.g.shape, device="cuda")
        gdr.gdr_bwd_dqkwg(p, dev(x.q), dev(x.k), dev(vn_r), dev(G_r), dev(hc_r), dev(dhc_r), dev(do), dev(dvn_r),
                          dq, dk_part, dw, dG_part, flags)
        gdr.gdr_bwd_wy(p, dev(x.k), dev(x.v), dev(x.beta), dev(G_r), dw, dev(dvn_r), dk_part, dG_part, dk, dv, dbeta,
                       dg, flags)
    torch.cuda.synchronize()
    tol = STAGE_TOL["bf16"]
    assert scaled_err(dq, a["dq"]) <= tol
    assert scaled_err(dk, a["dk"] + y["dk"]) <= tol
    assert scaled_err(dv, y["dv"]) <= tol
    assert scaled_err(dbeta, y["dbeta"]) <= tol
    assert scaled_err(dg, cb.reverse_cumsum(a["dG"] + y["dG"], C, per_k)) <= tol


# ---------------------------------------------------------------- grouped value heads

GROUPED = [(1, 128, 2, 2, 64, 64, 64), (2, 100, 1, 2, 128, 128, 64), (1, 96, 1, 3, 64, 128, 32)]


@pytest.mark.parametrize("shape", GROUPED, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("variant,dtype,per_k", [("simt", torch.float32, False), ("simt", torch.float32, True),
                                                  ("tensor", torch.bfloat16, False), ("tensor", torch.bfloat16, True)])
def test_grouped_value_heads_backward(shape, variant, dtype, per_k):
    B, T, H, G, K, V, C = shape
    x = grouped_inputs(B, T, H, G, K, V, per_k_gate=per_k, io_dtype=dtype, seed=80)
    do, dhf = upstream(x, 81)
    got, ran = gpu_backward(x, do, dhf, C, variant)
    assert ran == variant and got["dq"].shape == x.q.shape
    ref = reference(x, do, dhf, C, 1.0 / np.sqrt(K))
    for name in GRADS:
        err = scaled_err(got[name], ref[name])
        assert np.isfinite(err) and err <= BWD_TOL[io_name(dtype)], f"{name}: {err:.3e}"


@pytest.mark.parametrize("shape", SHAPES[:5], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("per_k", [False, True])
def test_fp16_io_backward(shape, per_k):
    B, T, H, K, V, C = shape
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=torch.float16, with_h0=True, seed=92)
    do, dhf = upstream(x, 93)
    got, ran = gpu_backward(x, do, dhf, C, "auto")
    assert ran == "simt" and got["dq"].dtype == torch.float16
    ref = reference(x, do, dhf, C, 1.0 / np.sqrt(K))
    for name in GRADS:
        err = scaled_err(got[name], ref[name])
        assert np.isfinite(err) and err <= BWD_TOL["f16"], f"{name}: {err:.3e}"


# ---------------------------------------------------------------- tensor-core local term and reverse scan

TC_SHAPES = [(2, 128, 3, 64, 64, 64), (1, 192, 2, 128, 128, 32), (2, 100, 2, 128, 64, 64), (1, 77, 1, 64, 128, 32)]


@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("per_k", [False, True])
def test_tensor_stage_dv_local(shape, per_k):
    x, do, _, full, _ = _stage_setup(shape, per_k, torch.bfloat16, 94)
    C = shape[-1]
    p = gdr.problem_for(x.q, x.v, x.g, C, scale=0.125, variant="tensor")
    G_r = rounded(full["G"], torch.float32)
    out = torch.full(x.v.shape, float("nan"), device="cuda", dtype=torch.bfloat16)
    gdr.gdr_bwd_dv_local_tc(p, dev(x.q), dev(x.k), dev(G_r), dev(do), out)
    torch.cuda.synchronize()
    assert scaled_err(out, cb.dv_local(x.q, x.k, G_r, do, C, 0.125)) <= STAGE_TOL["bf16"]


@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("per_k", [False, True])
def test_tensor_stage_reverse_scan_from_dv_local(shape, per_k):
    x, do, dhf, full, _ = _stage_setup(shape, per_k, torch.bfloat16, 96)
    B, T, H, K, V, C = shape
    p = gdr.problem_for(x.q, x.v, x.g, C, scale=0.125, variant="tensor")
    G_r, w_r = rounded(full["G"], torch.float32), rounded(full["w"], torch.bfloat16)
    dl_r = rounded(cb.dv_local(x.q, x.k, G_r, do, C, 0.125), torch.bfloat16)
    ref = cb.scan_dh(x.q, x.k, w_r, G_r, do, dl_r, dhf, C, 0.125)
    NT = -(-T // C)
    nan = float("nan")
    dh_ckpt = torch.full((B, NT, H, K, V), nan, device="cuda", dtype=torch.bfloat16)
    dv_new = torch.full((B, T, H, V), nan, device="cuda", dtype=torch.bfloat16)
    dh0 = torch.full((B, H, K, V), nan, device="cuda")
    gdr.gdr_bwd_scan_dh_tc(p, dev(x.q), dev(x.k), dev(w_r), dev(G_r), dev(dl_r), dev(do), dev(dhf), dh_ckpt, dv_new,
                           dh0)
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    tol = STAGE_TOL["bf16"]
    assert scaled_err(dh_ckpt, ref["dh_ckpt"]) <= tol
    assert scaled_err(dv_new, ref["dv_new"]) <= tol
    assert scaled_err(dh0, ref["dh0"]) <= tol


@pytest.mark.parametrize("shape", [(2, 128, 3, 64, 64, 32), (1, 96, 2, 128, 128, 32), (1, 77, 2, 128, 64, 32)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tensor_stage_wy_dqkg_at_32_token_chunks(shape):
    # the same per-chunk stage at C = 32 (two 16-row blocks, warps sharing the columns four ways)
    _wy_dqkg_case(shape)


KDA_STAGE_SHAPES = [(2, 128, 3, 64, 64, 64), (1, 192, 2, 128, 128, 64), (2, 100, 2, 128, 64, 64),
                    (1, 256, 1, 64, 128, 64), (2, 128, 3, 64, 64, 32), (1, 96, 2, 128, 128, 32),
                    (1, 77, 2, 128, 64, 32)]


@pytest.mark.parametrize("shape", KDA_STAGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_tensor_stage_wy_dqkg_per_key_gate(shape):
    # the per-key-dim gate's per-chunk stage: split-gate tiles around each chunk's middle row
    _wy_dqkg_case(shape, per_k=True)


@pytest.mark.parametrize("shape", KDA_STAGE_SHAPES[:3] + KDA_STAGE_SHAPES[5:], ids=lambda s: "x".join(map(str, s)))
def test_tensor_stage_wy_dqkg_per_key_gate_flagged_chunks(shape):
    # one head decays too fast for the split-gate products: its chunks are flagged and finished
    # by the CUDA-core stages, the other heads' chunks are not touched by them
    _wy_dqkg_case(shape, per_k=True, strong_head=0)


@pytest.mark.parametrize("shape", [(1, 128, 3, 64, 64, 64), (2, 100, 2, 128, 128, 32)],
                         ids=lambda s: "x".join(map(str, s)))
def test_backward_per_key_gate_mixed_spread(shape):
    # gdr_backward end to end with one head's chunks on the exact stages and the rest on the tensor cores
    B, T, H, K, V, C = shape
    x = make_inputs(B, T, H, K, V, per_k_gate=True, io_dtype=torch.bfloat16, with_h0=True, seed=98)
    g = x.g.clone()
    g[:, :, 1] *= 100.0
    x = GdrInputs(q=x.q, k=x.k, v=x.v, g=g, beta=x.beta, h0=x.h0 * 20)
    do, dhf = upstream(x, 99)
    got, ran = gpu_backward(x, do, dhf, C, "tensor")
    assert ran == "tensor"
    ref = reference(x, do, dhf, C, 1.0 / np.sqrt(K))
    for name in GRADS:
        err = scaled_err(got[name], ref[name])
        assert np.isfinite(err) and err <= BWD_TOL["bf16"], f"{name}: {err:.3e}"


def test_wy_dqkg_per_key_gate_needs_its_flags():
    x = make_inputs(1, 64, 1, 64, 64, per_k_gate=True, io_dtype=torch.bfloat16, seed=100)
    p = gdr.problem_for(x.q, x.v, x.g, 64, variant="tensor")
    t = torch.zeros(64, 1, 64, device="cuda", dtype=torch.bfloat16)
    gf = torch.zeros(1, 64, 1, 64, device="cuda")
    with pytest.raises(gdr.GdrError) as e:
        gdr.gdr_bwd_wy_dqkg(p, t, t, t, t, gf, t, t, t, t, t, t, t, t, t, t, t, t, gf, None)
    assert e.value.status == 1
