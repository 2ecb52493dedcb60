"""The segment-parallel scan on the GPU: the transfer scan and the stitch against
the segment-map oracle (oracle/segments.py), and gdr_forward with segments
against the token-recurrence oracle at the whole-forward bars.

Tolerances.  M and Z come from the tensor-core scan kernel run from the
identity and from zero: the bf16 checkpoint class, compared as relative
Frobenius error <= 1e-2 (the h_final bar).  The stitch is fp32 FMAs over K
terms per step: max |x - ref| / max |ref| <= 1e-5.  Whole forwards: the
forward's bars (bf16: o max-abs <= 2e-2, h_final rel-F <= 1e-2).
"""
import numpy as np
import pytest
import torch

from oracle import chunked, segments
from chunked_gated_delta_prepare_gb300 import gdr
from chunked_gated_delta_prepare_gb300.inputs import make_inputs
from gpu_helpers import H_TOL, STAGE_TOL, all_pairs, check_forward, dev, gpu_forward, grouped_inputs, rel_frob, \
    scaled_err

pytestmark = pytest.mark.gpu

# (B, T, H, K, V, C, S)
TRANSFER_CASES = [(1, 1024, 2, 128, 128, 64, 4), (2, 512, 3, 64, 64, 32, 4), (1, 768, 2, 64, 128, 64, 3),
                  (1, 512, 2, 128, 64, 32, 8), (2, 256, 1, 128, 128, 64, 1)]


def _rounded(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype)


@pytest.mark.parametrize("case", TRANSFER_CASES, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("per_k", [False, True])
def test_transfer_scan(case, per_k):
    B, T, H, K, V, C, S = case
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=torch.bfloat16, seed=110)
    p = chunked.prepare_wy(x.k, x.v, x.g, x.beta, C)
    w_r, u_r = _rounded(p["w"], torch.bfloat16), _rounded(p["u"], torch.bfloat16)
    G_r = _rounded(p["G"], torch.float32)
    M_ref, Z_ref = segments.segment_maps(x.k.double().numpy(), w_r.double().numpy(), u_r.double().numpy(),
                                         G_r.double().numpy(), C, S)
    prob = gdr.problem_for(x.q, x.v, x.g, C, variant="tensor")
    M = torch.full((B, S, H, K, K), float("nan"), device="cuda")
    Z = torch.full((B, S, H, K, V), float("nan"), device="cuda")
    gdr.gdr_scan_transfer(prob, dev(x.k), dev(w_r), dev(u_r), dev(G_r), S, M, Z)
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    assert rel_frob(M, M_ref) <= H_TOL["bf16"]
    assert rel_frob(Z, Z_ref) <= H_TOL["bf16"]


def test_transfer_scan_with_grouped_value_heads():
    B, T, H, G, K, V, C, S = 1, 512, 1, 2, 128, 128, 64, 2
    x = grouped_inputs(B, T, H, G, K, V, seed=111)
    p = chunked.prepare_wy(x.k, x.v, x.g, x.beta, C)
    w_r, u_r = _rounded(p["w"], torch.bfloat16), _rounded(p["u"], torch.bfloat16)
    G_r = _rounded(p["G"], torch.float32)
    M_ref, Z_ref = segments.segment_maps(x.k.double().numpy(), w_r.double().numpy(), u_r.double().numpy(),
                                         G_r.double().numpy(), C, S)
    prob = gdr.problem_for(x.q, x.v, x.g, C, variant="tensor")
    M = torch.full((B, S, H * G, K, K), float("nan"), device="cuda")
    Z = torch.full((B, S, H * G, K, V), float("nan"), device="cuda")
    gdr.gdr_scan_transfer(prob, dev(x.k), dev(w_r), dev(u_r), dev(G_r), S, M, Z)
    torch.cuda.synchronize()
    assert rel_frob(M, M_ref) <= H_TOL["bf16"] and rel_frob(Z, Z_ref) <= H_TOL["bf16"]


@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("with_h0", [False, True])
def test_stitch(K, V, with_h0):
    B, H, S = 2, 3, 5
    rng = np.random.default_rng(112)
    M = np.eye(K) * 0.9 + rng.standard_normal((B, S, H, K, K)) * 0.05
    Z = rng.standard_normal((B, S, H, K, V))
    h0 = rng.standard_normal((B, H, K, V)) if with_h0 else None
    starts_ref, hf_ref = segments.stitch(M, Z, h0)
    prob = gdr.make_problem(B, 64 * S, H, K, V, 64, torch.bfloat16)
    starts = torch.full((B, S, H, K, V), float("nan"), device="cuda")
    hf = torch.full((B, H, K, V), float("nan"), device="cuda")
    f32 = lambda a: None if a is None else torch.from_numpy(a).float().cuda()
    gdr.gdr_scan_combine(prob, S, f32(M), f32(Z), f32(h0), starts, hf)
    torch.cuda.synchronize()
    assert scaled_err(starts, starts_ref) <= STAGE_TOL["f32"]
    assert scaled_err(hf, hf_ref) <= STAGE_TOL["f32"]


# whole forwards with explicit segments: (B, T, H, K, V, C, S, per_k, variant)
FORWARD_CASES = [(1, 2048, 2, 128, 128, 64, 4, False, "fused"), (1, 2048, 2, 128, 128, 64, 8, False, "fused"),
                 (1, 2048, 2, 128, 128, 64, 4, False, "fused_tc"),
                 (2, 1024, 1, 64, 64, 64, 2, False, "fused"), (1, 2048, 2, 128, 128, 64, 4, True, "tensor"),
                 (1, 1024, 2, 64, 128, 32, 4, False, "tensor"), (2, 1024, 1, 128, 64, 32, 8, True, "tensor")]


@pytest.mark.parametrize("case", FORWARD_CASES, ids=lambda c: "x".join(map(str, c[:7])) + f"-{c[8]}-"
                         + ("kda" if c[7] else "gdn"))
def test_segmented_forward(case):
    B, T, H, K, V, C, S, per_k, variant = case
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=torch.bfloat16, with_h0=True, seed=113)
    p = gdr.problem_for(x.q, x.v, x.g, C, variant=variant, segments=S)
    assert gdr.gdr_forward_segments(p) == S
    o, hf, ran = gpu_forward(x, C, variant, segments=S)
    assert ran == variant
    check_forward(x, o, hf, all_pairs(B, H), C, 1.0 / np.sqrt(K), "bf16")
    o1, hf1, _ = gpu_forward(x, C, variant, segments=1)      # the serial scan: the same up to rounding
    assert (o.float() - o1.float()).abs().max().item() <= 2e-2
    assert rel_frob(hf, hf1.double().cpu().numpy()) <= 1e-2


def test_segmented_forward_with_grouped_heads_and_no_h0():
    x = grouped_inputs(1, 2048, 1, 2, 128, 128, with_h0=False, seed=114)
    o, hf, _ = gpu_forward(x, 64, "fused", segments=4)
    check_forward(x, o, hf, all_pairs(1, 2), 64, 1.0 / np.sqrt(128), "bf16")


def test_automatic_segments_forward():
    # one sequence and one head: 4 CTAs of serial scan, so the library cuts the 32 chunks in two
    x = make_inputs(1, 2048, 1, 128, 128, io_dtype=torch.bfloat16, with_h0=True, seed=115)
    assert gdr.gdr_forward_segments(gdr.problem_for(x.q, x.v, x.g, 64)) == 2
    o, hf, ran = gpu_forward(x, 64)
    assert ran == "fused"
    check_forward(x, o, hf, all_pairs(1, 1), 64, 1.0 / np.sqrt(128), "bf16")


def test_segment_arguments_are_checked():
    x = make_inputs(1, 2048, 1, 128, 128, io_dtype=torch.bfloat16, seed=116)
    for bad in (3, 64):
        p = gdr.problem_for(x.q, x.v, x.g, 64, segments=bad)
        assert gdr.gdr_forward_segments(p) == 0          # 3 and 64 do not divide the 32 chunks
    t = torch.zeros(1, 2048, 1, 128, device="cuda", dtype=torch.bfloat16)
    gf = torch.zeros(1, 2048, 1, device="cuda")
    m = torch.zeros(1, 3, 1, 128, 128, device="cuda")
    with pytest.raises(gdr.GdrError) as e:
        gdr.gdr_scan_transfer(gdr.problem_for(x.q, x.v, x.g, 64), t, t, t, gf, 3, m, m)
    assert e.value.status == 9


def test_low_head_count_workload_full_size():
    # the 32k-token sequence with 4 heads: the library picks 8 segments; two heads checked on every token
    from chunked_gated_delta_prepare_gb300 import workloads
    from chunked_gated_delta_prepare_gb300.inputs import make_workload_inputs
    wl = workloads.GDN_BF16_T32K_H4
    x = make_workload_inputs(wl)
    assert gdr.gdr_forward_segments(gdr.problem_for(x.q, x.v, x.g, wl.chunk)) == 8
    o, hf, ran = gpu_forward(x, wl.chunk)
    assert ran == "fused" and torch.isfinite(o).all() and torch.isfinite(hf).all()
    check_forward(x, o, hf, [(0, 0), (0, 3)], wl.chunk, 1.0 / np.sqrt(wl.K), wl.io)


# ---------------------------------------------------------------- the backward's segments

@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (128, 64)])
@pytest.mark.parametrize("with_dhf", [False, True])
def test_reverse_stitch(K, V, with_dhf):
    B, H, S = 2, 2, 6
    rng = np.random.default_rng(120)
    M = np.eye(K) * 0.9 + rng.standard_normal((B, S, H, K, K)) * 0.05
    Zb = rng.standard_normal((B, S, H, K, V))
    dhf = rng.standard_normal((B, H, K, V)) if with_dhf else None
    ends_ref, dh0_ref = segments.stitch_reverse(M, Zb, dhf)
    prob = gdr.make_problem(B, 64 * S, H, K, V, 64, torch.bfloat16)
    ends = torch.full((B, S, H, K, V), float("nan"), device="cuda")
    dh0 = torch.full((B, H, K, V), float("nan"), device="cuda")
    f32 = lambda a: None if a is None else torch.from_numpy(a).float().cuda()
    gdr.gdr_scan_combine_reverse(prob, S, f32(M), f32(Zb), f32(dhf), ends, dh0)
    torch.cuda.synchronize()
    assert scaled_err(ends, ends_ref) <= STAGE_TOL["f32"]
    assert scaled_err(dh0, dh0_ref) <= STAGE_TOL["f32"]


# (B, T, H, K, V, C, S, per_k): the scalar gate at C = 64 (local term from P) and C = 32 (its own
# kernel), the per-key gate (exactly flagged chunks included by the strong-decay case below)
BACKWARD_CASES = [(1, 2048, 2, 128, 128, 64, 4, False), (2, 1024, 1, 64, 64, 64, 8, False),
                  (1, 1024, 2, 64, 128, 32, 4, False), (1, 2048, 2, 128, 128, 64, 4, True),
                  (2, 1024, 1, 128, 64, 32, 2, True)]


@pytest.mark.parametrize("case", BACKWARD_CASES, ids=lambda c: "x".join(map(str, c[:7])) + ("-kda" if c[7] else "-gdn"))
def test_segmented_backward(case):
    from test_gpu_backward import BWD_TOL, GRADS, gpu_backward, reference, upstream
    B, T, H, K, V, C, S, per_k = case
    x = make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=torch.bfloat16, with_h0=True, seed=121)
    do, dhf = upstream(x, 122)
    assert gdr.gdr_forward_segments(gdr.problem_for(x.q, x.v, x.g, C, variant="tensor", segments=S)) == S
    got, ran = gpu_backward(x, do, dhf, C, "tensor", segments=S)
    assert ran == "tensor"
    ref = reference(x, do, dhf, C, 1.0 / np.sqrt(K))
    for name in GRADS:
        err = scaled_err(got[name], ref[name])
        assert np.isfinite(err) and err <= BWD_TOL["bf16"], f"{name}: {err:.3e}"


def test_segmented_backward_grouped_heads_strong_decay_and_no_final_gradient():
    from test_gpu_backward import BWD_TOL, GRADS, gpu_backward, reference, upstream
    from chunked_gated_delta_prepare_gb300.inputs import GdrInputs
    x = grouped_inputs(1, 2048, 1, 2, 128, 128, per_k_gate=True, seed=123)
    g = x.g.clone()
    g[:, :, 1] *= 100.0                 # the second value head's chunks go to the exact per-chunk stages
    x = GdrInputs(q=x.q, k=x.k, v=x.v, g=g, beta=x.beta, h0=x.h0)
    do, _ = upstream(x, 124)
    got, _ = gpu_backward(x, do, None, 64, "tensor", segments=4)
    ref = reference(x, do, None, 64, 1.0 / np.sqrt(128))
    for name in GRADS:
        err = scaled_err(got[name], ref[name])
        assert np.isfinite(err) and err <= BWD_TOL["bf16"], f"{name}: {err:.3e}"


def test_automatic_segments_backward():
    from test_gpu_backward import BWD_TOL, GRADS, gpu_backward, reference, upstream
    x = make_inputs(1, 2048, 1, 128, 128, io_dtype=torch.bfloat16, with_h0=True, seed=125)
    do, dhf = upstream(x, 126)
    got, _ = gpu_backward(x, do, dhf, 64, "auto")
    ref = reference(x, do, dhf, 64, 1.0 / np.sqrt(128))
    for name in GRADS:
        assert scaled_err(got[name], ref[name]) <= BWD_TOL["bf16"], name
