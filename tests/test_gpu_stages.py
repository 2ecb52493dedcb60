"""Per-stage parity on the GPU: each C-ABI stage entry point against the
chunked float64 oracle's stage function, fed the same rounded inputs."""
import itertools

import numpy as np
import pytest
import torch

from oracle import chunked
from chunked_gated_delta_prepare_gb300 import gdr
from chunked_gated_delta_prepare_gb300.inputs import make_inputs
from gpu_helpers import STAGE_TOL, dev, io_name, rel_frob, scaled_err

pytestmark = pytest.mark.gpu

# (B, T, H, K, V, C): several chunks per head, odd head counts, K != V, both chunk sizes
SHAPES = [(2, 256, 3, 64, 64, 64), (1, 192, 2, 128, 128, 64), (2, 128, 3, 64, 128, 32),
          (1, 160, 1, 128, 64, 32), (1, 256, 2, 128, 128, 32), (2, 128, 1, 64, 64, 32),
          # a last, partial chunk (T not a multiple of C)
          (2, 100, 3, 64, 64, 64), (1, 77, 2, 128, 128, 32), (1, 20, 1, 128, 64, 64)]
# per stage: the variants that run it, with the io dtypes each one takes
BOTH = (torch.float32, torch.bfloat16)
IO16 = (torch.bfloat16, torch.float16)
STAGE_VARIANTS = {
    "prepare": {"simt": BOTH, "tensor": IO16},
    "scan": {"simt": BOTH, "tensor": IO16},
    "output": {"simt": BOTH, "tensor": IO16},
}


def cases(stage):
    for shape, per_k, (variant, dtypes) in itertools.product(SHAPES, (False, True), STAGE_VARIANTS[stage].items()):
        for dt in dtypes:
            yield pytest.param(shape, per_k, variant, dt,
                               id=f"{'x'.join(map(str, shape))}-{'kda' if per_k else 'gdn'}-{variant}-{io_name(dt)}")


@pytest.mark.parametrize("stage", ["prepare", "scan", "output"])
def test_tensor_variant_refuses_fp32(stage):
    x = make_inputs(1, 64, 1, 64, 64, io_dtype=torch.float32)
    p = gdr.problem_for(x.q, x.v, x.g, 64, variant="tensor")
    t = torch.zeros(64, 1, 64, device="cuda")
    with pytest.raises(gdr.GdrError) as e:
        if stage == "prepare":
            gdr.gdr_prepare_wy(p, t, t, t, t, t, t, t)
        elif stage == "scan":
            gdr.gdr_scan_h(p, t, t, t, t, None, None, t, None)
        else:
            gdr.gdr_chunk_output(p, t, t, t, t, t, t)
    assert e.value.status == 8


def rounded(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype)


@pytest.mark.parametrize("shape,per_k,variant,dtype", list(cases("prepare")))
def test_prepare_stage(shape, per_k, variant, dtype):
    B, T, H, K, V, C = shape
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=dtype, with_h0=False, seed=1)
    p = gdr.problem_for(x.q, x.v, x.g, C, variant=variant)
    k, v, g, beta = (dev(t) for t in (x.k, x.v, x.g, x.beta))
    w = torch.full_like(k, float("nan"))
    u = torch.full_like(v, float("nan"))
    g_cum = torch.full_like(g, float("nan"))
    gdr.gdr_prepare_wy(p, k, v, g, beta, w, u, g_cum)
    torch.cuda.synchronize()
    assert gdr.gdr_last_variant() == variant
    ref = chunked.prepare_wy(x.k, x.v, x.g, x.beta, C)
    io = io_name(dtype)
    assert scaled_err(g_cum, ref["G"]) <= 1e-6
    assert scaled_err(w, ref["w"]) <= STAGE_TOL[io]
    assert scaled_err(u, ref["u"]) <= STAGE_TOL[io]


@pytest.mark.parametrize("shape,per_k,variant,dtype", list(cases("scan")))
@pytest.mark.parametrize("with_h0", [False, True])
def test_scan_stage(shape, per_k, variant, dtype, with_h0):
    B, T, H, K, V, C = shape
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=dtype, with_h0=with_h0, seed=2)
    pre = chunked.prepare_wy(x.k, x.v, x.g, x.beta, C)
    w_r, u_r = rounded(pre["w"], dtype), rounded(pre["u"], dtype)
    G_r = rounded(pre["G"], torch.float32)
    h0 = None if x.h0 is None else x.h0 * 20          # a state large enough to matter
    ref = chunked.scan_h(x.k, w_r, u_r, G_r, h0, C)
    p = gdr.problem_for(x.q, x.v, x.g, C, variant=variant)
    NT = -(-T // C)
    h_ckpt = torch.full((B, NT, H, K, V), float("nan"), device="cuda", dtype=dtype)
    v_new = torch.full((B, T, H, V), float("nan"), device="cuda", dtype=dtype)
    h_final = torch.full((B, H, K, V), float("nan"), device="cuda", dtype=torch.float32)
    gdr.gdr_scan_h(p, dev(x.k), dev(w_r), dev(u_r), dev(G_r), dev(h0), h_ckpt, v_new, h_final)
    torch.cuda.synchronize()
    assert gdr.gdr_last_variant() == variant
    io = io_name(dtype)
    assert scaled_err(v_new, ref["v_new"]) <= STAGE_TOL[io]
    assert scaled_err(h_ckpt, ref["ckpt"]) <= STAGE_TOL[io]
    assert rel_frob(h_final, ref["h_final"]) <= STAGE_TOL[io]
    if h0 is None:
        assert float(h_ckpt[:, 0].abs().max()) == 0.0
    else:
        assert scaled_err(h_ckpt[:, 0], h0.numpy()) <= STAGE_TOL[io]


@pytest.mark.parametrize("shape,per_k,variant,dtype", list(cases("scan")))
def test_scan_stage_optional_outputs(shape, per_k, variant, dtype):
    """h_ckpt and h_final may be NULL; v_new must not change when they are."""
    B, T, H, K, V, C = shape
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=dtype, with_h0=True, seed=3)
    pre = chunked.prepare_wy(x.k, x.v, x.g, x.beta, C)
    w_r, u_r, G_r = rounded(pre["w"], dtype), rounded(pre["u"], dtype), rounded(pre["G"], torch.float32)
    p = gdr.problem_for(x.q, x.v, x.g, C, variant=variant)
    args = (dev(x.k), dev(w_r), dev(u_r), dev(G_r), dev(x.h0))
    v1 = torch.empty(B, T, H, V, device="cuda", dtype=dtype)
    v2 = torch.empty_like(v1)
    hc = torch.empty(B, -(-T // C), H, K, V, device="cuda", dtype=dtype)
    hf = torch.empty(B, H, K, V, device="cuda", dtype=torch.float32)
    gdr.gdr_scan_h(p, *args, hc, v1, hf)
    gdr.gdr_scan_h(p, *args, None, v2, None)
    torch.cuda.synchronize()
    assert torch.equal(v1, v2)


@pytest.mark.parametrize("shape,per_k,variant,dtype", list(cases("output")))
def test_output_stage(shape, per_k, variant, dtype):
    B, T, H, K, V, C = shape
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=dtype, with_h0=True, seed=4)
    full = chunked.forward_chunked(x.q, x.k, x.v, x.g, x.beta, x.h0 * 20, C, 0.125)
    vn_r, ck_r = rounded(full["v_new"], dtype), rounded(full["ckpt"], dtype)
    G_r = rounded(full["G"], torch.float32)
    ref = chunked.chunk_output(x.q, x.k, vn_r, ck_r, G_r, C, 0.125)
    p = gdr.problem_for(x.q, x.v, x.g, C, scale=0.125, variant=variant)
    o = torch.full((B, T, H, V), float("nan"), device="cuda", dtype=dtype)
    gdr.gdr_chunk_output(p, dev(x.q), dev(x.k), dev(vn_r), dev(ck_r), dev(G_r), o)
    torch.cuda.synchronize()
    assert gdr.gdr_last_variant() == variant
    assert scaled_err(o, ref) <= STAGE_TOL[io_name(dtype)]


SCAN_OUTPUT_SHAPES = [(2, 256, 3, 64, 64, 64), (1, 192, 2, 128, 128, 64), (2, 128, 3, 64, 128, 32),
                      (1, 160, 1, 128, 64, 32), (1, 64, 2, 128, 128, 64), (2, 100, 3, 64, 64, 64),
                      (1, 77, 1, 128, 128, 32)]


@pytest.mark.parametrize("shape", SCAN_OUTPUT_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("with_h0", [False, True])
@pytest.mark.parametrize("dtype", IO16, ids=io_name)
def test_scan_output_stage(shape, with_h0, dtype):
    """Scan and output fused: o and h_final against the chunked oracle's scan and
    output stages fed the same rounded w, u, G."""
    B, T, H, K, V, C = shape
    x = make_inputs(B, T, H, K, V, io_dtype=dtype, with_h0=with_h0, seed=14)
    pre = chunked.prepare_wy(x.k, x.v, x.g, x.beta, C)
    w_r, u_r, G_r = rounded(pre["w"], dtype), rounded(pre["u"], dtype), rounded(pre["G"], torch.float32)
    h0 = None if x.h0 is None else x.h0 * 20
    scan = chunked.scan_h(x.k, w_r, u_r, G_r, h0, C)
    o_ref = chunked.chunk_output(x.q, x.k, scan["v_new"], scan["ckpt"], G_r, C, 0.125)
    p = gdr.problem_for(x.q, x.v, x.g, C, scale=0.125)
    o = torch.full((B, T, H, V), float("nan"), device="cuda", dtype=dtype)
    hf = torch.full((B, H, K, V), float("nan"), device="cuda", dtype=torch.float32)
    gdr.gdr_scan_output(p, dev(x.q), dev(x.k), dev(w_r), dev(u_r), dev(G_r), None, dev(h0), o, hf)
    torch.cuda.synchronize()
    assert gdr.gdr_last_variant() == "fused" and o.dtype == dtype
    assert scaled_err(o, o_ref) <= STAGE_TOL[io_name(dtype)]
    assert rel_frob(hf, scan["h_final"]) <= STAGE_TOL[io_name(dtype)]


@pytest.mark.parametrize("shape", [(2, 256, 3, 128, 128, 64), (1, 100, 2, 128, 128, 64), (1, 64, 1, 128, 128, 64)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("with_h0", [False, True])
def test_scan_output_stage_tcgen05(shape, with_h0):
    """The tcgen05 form of the fused scan and output (variant FUSED_TC), fed the oracle's rounded w, u, G
    and gated scores P, against the chunked oracle's scan and output stages."""
    B, T, H, K, V, C = shape
    dtype = torch.bfloat16
    x = make_inputs(B, T, H, K, V, io_dtype=dtype, with_h0=with_h0, seed=15)
    pre = chunked.prepare_wy(x.k, x.v, x.g, x.beta, C)
    w_r, u_r, G_r = rounded(pre["w"], dtype), rounded(pre["u"], dtype), rounded(pre["G"], torch.float32)
    P_r = rounded(chunked.gated_causal_scores(x.q, x.k, G_r, C), dtype)
    h0 = None if x.h0 is None else x.h0 * 20
    scan = chunked.scan_h(x.k, w_r, u_r, G_r, h0, C)
    o_ref = chunked.chunk_output(x.q, x.k, scan["v_new"], scan["ckpt"], G_r, C, 0.125)
    p = gdr.problem_for(x.q, x.v, x.g, C, scale=0.125, variant="fused_tc")
    o = torch.full((B, T, H, V), float("nan"), device="cuda", dtype=dtype)
    hf = torch.full((B, H, K, V), float("nan"), device="cuda", dtype=torch.float32)
    gdr.gdr_scan_output(p, dev(x.q), dev(x.k), dev(w_r), dev(u_r), dev(G_r), dev(P_r), dev(h0), o, hf)
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    assert gdr.gdr_last_variant() == "fused_tc"
    assert scaled_err(o, o_ref) <= STAGE_TOL["bf16"]
    assert rel_frob(hf, scan["h_final"]) <= STAGE_TOL["bf16"]


def _gated_ref(x, G, C):
    """qg = q exp(G) and kg = k exp(G_last - G) per chunk (G_last the chunk's last token, or the last
    one before T), from their definitions on the oracle's G."""
    q, k, G = (t.double().numpy() for t in (x.q, x.k, G))
    T = q.shape[1]
    qg, kg = q * np.exp(G), np.empty_like(k)
    for t0 in range(0, T, C):
        t1 = min(T, t0 + C)
        kg[:, t0:t1] = k[:, t0:t1] * np.exp(G[:, t1 - 1:t1] - G[:, t0:t1])
    return qg, kg


@pytest.mark.parametrize("shape", [(1, 256, 2, 128, 128, 64), (2, 100, 1, 128, 128, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gated_operands_stage(shape):
    """gdr_gated_operands (per-key-dim gate) on the oracle's rounded G: P against the chunked oracle's
    gated scores, qg and kg against their definitions."""
    B, T, H, K, V, C = shape
    x = make_inputs(B, T, H, K, V, per_k_gate=True, io_dtype=torch.bfloat16, seed=16)
    G_r = rounded(chunked.prepare_wy(x.k, x.v, x.g, x.beta, C)["G"], torch.float32)
    NT = -(-T // C)
    P = torch.full((B, NT, H, C, C), float("nan"), device="cuda", dtype=torch.bfloat16)
    kg = torch.full((B, T, H, K), float("nan"), device="cuda", dtype=torch.bfloat16)
    qg = torch.full((B, T, H, K), float("nan"), device="cuda", dtype=torch.bfloat16)
    p = gdr.problem_for(x.q, x.v, x.g, C)
    gdr.gdr_gated_operands(p, dev(x.q), dev(x.k), dev(G_r), P, kg, qg)
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    qg_ref, kg_ref = _gated_ref(x, G_r, C)
    assert scaled_err(P, chunked.gated_causal_scores(x.q, x.k, G_r, C)) <= STAGE_TOL["bf16"]
    assert scaled_err(qg, qg_ref) <= STAGE_TOL["bf16"] and scaled_err(kg, kg_ref) <= STAGE_TOL["bf16"]


@pytest.mark.parametrize("shape", [(1, 256, 2, 128, 128, 64), (2, 100, 1, 128, 128, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_scan_output_stage_tcgen05_per_key_gate(shape):
    """The tcgen05 scan and output with a per-key-dim gate, fed the oracle's rounded w, u, G, P, qg and kg,
    against the chunked oracle's scan and output stages."""
    B, T, H, K, V, C = shape
    dtype = torch.bfloat16
    x = make_inputs(B, T, H, K, V, per_k_gate=True, io_dtype=dtype, with_h0=True, seed=17)
    pre = chunked.prepare_wy(x.k, x.v, x.g, x.beta, C)
    w_r, u_r, G_r = rounded(pre["w"], dtype), rounded(pre["u"], dtype), rounded(pre["G"], torch.float32)
    P_r = rounded(chunked.gated_causal_scores(x.q, x.k, G_r, C), dtype)
    qg_ref, kg_ref = _gated_ref(x, G_r, C)
    qg_r, kg_r = rounded(qg_ref, dtype), rounded(kg_ref, dtype)
    h0 = x.h0 * 20
    scan = chunked.scan_h(x.k, w_r, u_r, G_r, h0, C)
    o_ref = chunked.chunk_output(x.q, x.k, scan["v_new"], scan["ckpt"], G_r, C, 0.125)
    p = gdr.problem_for(x.q, x.v, x.g, C, scale=0.125, variant="fused_tc")
    o = torch.full((B, T, H, V), float("nan"), device="cuda", dtype=dtype)
    hf = torch.full((B, H, K, V), float("nan"), device="cuda", dtype=torch.float32)
    gdr.gdr_scan_output(p, dev(qg_r), dev(kg_r), dev(w_r), dev(u_r), dev(G_r), dev(P_r), dev(h0), o, hf)
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0 and gdr.gdr_last_variant() == "fused_tc"
    assert scaled_err(o, o_ref) <= STAGE_TOL["bf16"]
    assert rel_frob(hf, scan["h_final"]) <= STAGE_TOL["bf16"]
    # the per-key-dim gate runs only on the tcgen05 kernel, with P
    p.variant = gdr.VARIANTS["auto"]
    with pytest.raises(gdr.GdrError) as e:
        gdr.gdr_scan_output(p, dev(qg_r), dev(kg_r), dev(w_r), dev(u_r), dev(G_r), dev(P_r), dev(h0), o, hf)
    assert e.value.status == 8


def test_scan_output_tcgen05_needs_the_scores():
    x = make_inputs(1, 64, 1, 128, 128, io_dtype=torch.bfloat16)
    t = torch.zeros(64, 1, 128, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(gdr.GdrError) as e:
        gdr.gdr_scan_output(gdr.problem_for(x.q, x.v, x.g, 64, variant="fused_tc"), t, t, t, t, t, None, None, t, None)
    assert e.value.status == 8


def test_scan_output_refuses_per_key_gate_and_fp32():
    x = make_inputs(1, 64, 1, 64, 64, per_k_gate=True, io_dtype=torch.bfloat16)
    t = torch.zeros(64, 1, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(gdr.GdrError) as e:
        gdr.gdr_scan_output(gdr.problem_for(x.q, x.v, x.g, 64), t, t, t, t, t, None, None, t, None)
    assert e.value.status == 8
    xf = make_inputs(1, 64, 1, 64, 64, io_dtype=torch.float32)
    tf = torch.zeros(64, 1, 64, device="cuda")
    with pytest.raises(gdr.GdrError) as e:
        gdr.gdr_scan_output(gdr.problem_for(xf.q, xf.v, xf.g, 64), tf, tf, tf, tf, tf, None, None, tf, None)
    assert e.value.status == 8


@pytest.mark.parametrize("shape", [(2, 256, 3, 64, 64, 64), (1, 192, 2, 128, 128, 64), (1, 320, 1, 128, 64, 64),
                                   (2, 100, 2, 128, 128, 64), (2, 20, 1, 64, 64, 64)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", IO16, ids=io_name)
def test_prepare_with_scores_then_scan_output(shape, dtype):
    """gdr_prepare_wyp's P against the oracle's gated causal scores, then
    gdr_scan_output reading that P against the oracle's scan and output."""
    B, T, H, K, V, C = shape
    x = make_inputs(B, T, H, K, V, io_dtype=dtype, with_h0=True, seed=15)
    p = gdr.problem_for(x.q, x.v, x.g, C, scale=0.125)
    q, k, v, g, beta = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta))
    NT = -(-T // C)
    w = torch.full_like(k, float("nan"))
    u = torch.full_like(v, float("nan"))
    g_cum = torch.full_like(g, float("nan"))
    P = torch.full((B, NT, H, C, C), float("nan"), device="cuda", dtype=dtype)
    gdr.gdr_prepare_wyp(p, q, k, v, g, beta, w, u, g_cum, P)
    torch.cuda.synchronize()
    pre = chunked.prepare_wy(x.k, x.v, x.g, x.beta, C)
    assert scaled_err(w, pre["w"]) <= STAGE_TOL[io_name(dtype)]
    assert scaled_err(u, pre["u"]) <= STAGE_TOL[io_name(dtype)]
    assert scaled_err(g_cum, pre["G"]) <= 1e-6
    assert scaled_err(P, chunked.gated_causal_scores(x.q, x.k, pre["G"], C)) <= STAGE_TOL[io_name(dtype)]
    o = torch.full((B, T, H, V), float("nan"), device="cuda", dtype=dtype)
    hf = torch.full((B, H, K, V), float("nan"), device="cuda", dtype=torch.float32)
    gdr.gdr_scan_output(p, q, k, w, u, g_cum, P, dev(x.h0), o, hf)
    torch.cuda.synchronize()
    w_r, u_r, G_r, P_r = w.cpu(), u.cpu(), g_cum.cpu(), P.cpu()
    scan = chunked.scan_h(x.k, w_r, u_r, G_r, x.h0, C)
    # the output with the GPU's P (rounded) in place of the oracle's scores
    # (a partial last chunk: zero q and v' past T, G held at its last value, then cut back to T)
    qc = chunked._to_chunks(chunked._pad_tokens(chunked._f64(x.q), C), C)
    vc = chunked._to_chunks(chunked._pad_tokens(scan["v_new"], C), C)
    Gc = chunked._gate_vec(chunked._pad_tokens(chunked._f64(G_r), C, edge=True), C)
    o_ref = chunked._from_chunks(0.125 * ((qc * np.exp(Gc)) @ scan["ckpt"] + chunked._f64(P_r) @ vc))[:, :T]
    assert scaled_err(o, o_ref) <= STAGE_TOL[io_name(dtype)]
    assert rel_frob(hf, scan["h_final"]) <= STAGE_TOL[io_name(dtype)]
