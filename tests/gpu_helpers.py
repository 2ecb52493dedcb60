"""Helpers shared by the GPU parity tests: run libgdr through its C ABI on
seeded inputs, run the oracle on the same rounded inputs, and compare.

Tolerances.  The whole-forward bars are the workloads' stated ones: for bf16 io,
max |o - o_ref| <= 2e-2 and ||h_final - h_ref||_F / ||h_ref||_F <= 1e-2; for fp32
io both <= 1e-4.  Per-stage outputs (w, u, v_new, checkpoints, g_cum, o of the
output stage alone) are compared as max|x - ref| / max|ref|: <= 1e-2 for bf16
(a bf16 store alone is a 2^-9 relative rounding, and the tensor-core operands are
bf16 too, with fp32 accumulation over at most 128 terms) and <= 1e-5 for fp32
(fp32 FMAs with at most a few hundred terms per sum).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import chunked
from chunked_gated_delta_prepare_gb300 import gdr

# fp16 io (10-bit mantissa, a 2^-11 relative step per stored value) meets the bf16 bars with room
O_TOL = {"bf16": 2e-2, "f16": 2e-2, "f32": 1e-4}
H_TOL = {"bf16": 1e-2, "f16": 1e-2, "f32": 1e-4}
STAGE_TOL = {"bf16": 1e-2, "f16": 1e-2, "f32": 1e-5}


def io_name(dtype):
    return {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[dtype]


def dev(t):
    return None if t is None else t.to("cuda").contiguous()


def scaled_err(x, ref):
    x = np.asarray(x.detach().to("cpu").double().numpy() if hasattr(x, "detach") else x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = max(np.abs(ref).max(), 1e-30)
    return float(np.abs(x - ref).max() / den)


def max_abs(x, ref):
    x = x.detach().to("cpu").double().numpy() if hasattr(x, "detach") else np.asarray(x)
    return float(np.abs(x - ref).max())


def rel_frob(x, ref):
    x = x.detach().to("cpu").double().numpy() if hasattr(x, "detach") else np.asarray(x)
    return float(np.linalg.norm((x - ref).ravel()) / max(np.linalg.norm(np.asarray(ref).ravel()), 1e-30))


def variant_supports(variant, K, V, C, per_k=False):
    """Whether a forward variant takes these sizes (the tcgen05 fused form: K = V = 128, C = 64, either gate;
    the warp-level fused form: a scalar gate)."""
    if variant == "fused_tc":
        return K == 128 and V == 128 and C == 64
    if variant == "fused":
        return not per_k
    return True


def problem(x, C, variant="auto", scale=None):
    return gdr.problem_for(x.q, x.v, x.g, C, scale, variant)


def gpu_forward(x, C, variant="auto", scale=None, want_h_final=True, h0="inputs", segments=0):
    """gdr_forward through the C ABI on device copies of the inputs."""
    q, k, v, g, beta = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta))
    h0d = dev(x.h0) if h0 == "inputs" else dev(h0)
    p = gdr.problem_for(q, v, g, C, scale, variant, segments)
    B, T, _, K = q.shape
    H, V = v.shape[2], v.shape[-1]            # value heads
    o = torch.full((B, T, H, V), float("nan"), device="cuda", dtype=q.dtype)
    hf = torch.full((B, H, K, V), float("nan"), device="cuda", dtype=torch.float32) if want_h_final else None
    nbytes = gdr.gdr_forward_workspace_bytes(p)
    ws = torch.empty(max(nbytes, 1), device="cuda", dtype=torch.uint8)
    gdr.gdr_forward(p, q, k, v, g, beta, h0d, o, hf, ws if nbytes else None, nbytes)
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    return o, hf, gdr.gdr_last_variant()


def sample_heads(x, pairs):
    """Slice the inputs down to the given (b, h) pairs of value heads, as a batch of single-head
    problems (with grouped value heads, value head h reads the q and k of head h // G)."""
    G = x.v.shape[2] // x.q.shape[2]

    def tokens(t):   # [B,T,H,...] -> [P,T,1,...]
        return torch.stack([t[b, :, h] for b, h in pairs]).unsqueeze(2)

    def qk(t):
        return torch.stack([t[b, :, h // G] for b, h in pairs]).unsqueeze(2)

    def state(t):    # [B,H,K,V] -> [P,1,K,V]
        return None if t is None else torch.stack([t[b, h] for b, h in pairs]).unsqueeze(1)
    return dict(q=qk(x.q), k=qk(x.k), v=tokens(x.v), g=tokens(x.g), beta=tokens(x.beta),
                h0=state(x.h0))


def oracle_heads(x, pairs, C, scale):
    """Token-recurrence oracle on the selected heads (all T tokens of each)."""
    s = sample_heads(x, pairs)
    return oracle.naive_forward(s["q"], s["k"], s["v"], s["g"], s["beta"], s["h0"], C, scale, with_ckpt=False)


def gather_heads(t, pairs, state=False):
    t = t.detach().to("cpu").double().numpy()
    if state:
        return np.stack([t[b, h] for b, h in pairs])[:, None]
    return np.stack([t[b, :, h] for b, h in pairs])[:, :, None]


def check_forward(x, o, hf, pairs, C, scale, io):
    ref = oracle_heads(x, pairs, C, scale)
    eo = max_abs(gather_heads(o, pairs), ref["o"])
    eh = rel_frob(gather_heads(hf, pairs, state=True), ref["h_final"]) if hf is not None else 0.0
    assert np.isfinite(eo) and eo <= O_TOL[io], f"o max-abs error {eo:.3e} > {O_TOL[io]}"
    assert np.isfinite(eh) and eh <= H_TOL[io], f"h_final rel-Frobenius error {eh:.3e} > {H_TOL[io]}"
    return eo, eh


def all_pairs(B, H):
    return [(b, h) for b in range(B) for h in range(H)]


def grouped_inputs(B, T, H, G, K, V, *, per_k_gate=False, io_dtype=torch.bfloat16, with_h0=True, seed=0):
    """Inputs with H q/k heads shared by H * G value heads (grouped value heads)."""
    from chunked_gated_delta_prepare_gb300.inputs import GdrInputs, make_inputs
    x = make_inputs(B, T, H * G, K, V, per_k_gate=per_k_gate, io_dtype=io_dtype, with_h0=with_h0, seed=seed)
    return GdrInputs(q=x.q[:, :, ::G].contiguous(), k=x.k[:, :, ::G].contiguous(), v=x.v, g=x.g, beta=x.beta,
                     h0=x.h0)
