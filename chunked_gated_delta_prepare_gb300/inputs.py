"""Seeded synthetic inputs for the chunked gated-delta-rule forward.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle.  It holds no arithmetic of the method itself: it only draws random
tensors and shapes them into the value distributions that the workloads use
(unit-norm queries and keys, standard-normal values, sigmoid betas,
logsigmoid/16 log-decays, an optional small initial state).

Draw order (fixed, one CPU generator seeded once):
    q, k ~ N(0,1) [B,T,H,K];  v ~ N(0,1) [B,T,H,V];  beta_logit ~ N(0,1) [B,T,H];
    g_logit ~ N(0,1) [B,T,H] (scalar gate) or [B,T,H,K] (per-key-dim gate);
    h0 ~ 0.02 * N(0,1) [B,H,K,V] when the workload has a non-zero initial state.
Then, in fp32: q, k are L2-normalised over the last dim, beta = sigmoid(beta_logit),
g = logsigmoid(g_logit) / 16.  q, k, v, beta are then rounded to the io dtype; g and
h0 stay fp32.  Every consumer (GPU or CPU) reads the same rounded values.

Packed variable-length batches (make_varlen_inputs) draw one sequence of all
the tokens the same way (B = 1, T = total, value heads), keep the first H heads
of q and k, and draw the n initial states afterwards from a second generator
(seed + 1); cu_seqlens is the running sum of the given lengths.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass
class GdrInputs:
    q: torch.Tensor        # [B,T,H,K] io dtype
    k: torch.Tensor        # [B,T,H,K] io dtype
    v: torch.Tensor        # [B,T,H,V] io dtype
    g: torch.Tensor        # [B,T,H] or [B,T,H,K] fp32, natural-log per-token decay
    beta: torch.Tensor     # [B,T,H] io dtype
    h0: torch.Tensor | None  # [B,H,K,V] fp32 or None (zero initial state)

    def tensors(self):
        return dict(q=self.q, k=self.k, v=self.v, g=self.g, beta=self.beta, h0=self.h0)


def make_inputs(B: int, T: int, H: int, K: int, V: int, *, per_k_gate: bool = False,
                io_dtype: torch.dtype = torch.bfloat16, with_h0: bool = False,
                seed: int = 0) -> GdrInputs:
    """Draw one seeded problem on the CPU (see the module docstring for the recipe)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    q = torch.randn(B, T, H, K, generator=gen, dtype=torch.float32)
    k = torch.randn(B, T, H, K, generator=gen, dtype=torch.float32)
    v = torch.randn(B, T, H, V, generator=gen, dtype=torch.float32)
    beta_logit = torch.randn(B, T, H, generator=gen, dtype=torch.float32)
    gshape = (B, T, H, K) if per_k_gate else (B, T, H)
    g_logit = torch.randn(*gshape, generator=gen, dtype=torch.float32)
    h0 = None
    if with_h0:
        h0 = 0.02 * torch.randn(B, H, K, V, generator=gen, dtype=torch.float32)
    q = q / q.norm(dim=-1, keepdim=True)
    k = k / k.norm(dim=-1, keepdim=True)
    beta = torch.sigmoid(beta_logit)
    g = torch.nn.functional.logsigmoid(g_logit) / 16.0
    return GdrInputs(q=q.to(io_dtype).contiguous(), k=k.to(io_dtype).contiguous(),
                     v=v.to(io_dtype).contiguous(), g=g.contiguous(),
                     beta=beta.to(io_dtype).contiguous(), h0=h0)


@dataclass
class VarlenInputs:
    q: torch.Tensor        # [total,H,K] io dtype
    k: torch.Tensor        # [total,H,K] io dtype
    v: torch.Tensor        # [total,HV,V] io dtype
    g: torch.Tensor        # [total,HV] or [total,HV,K] fp32
    beta: torch.Tensor     # [total,HV] io dtype
    h0: torch.Tensor | None  # [n,HV,K,V] fp32 or None
    cu: torch.Tensor       # [n + 1] int32: sequence s holds the rows cu[s] .. cu[s+1]-1

    def tensors(self):
        return dict(q=self.q, k=self.k, v=self.v, g=self.g, beta=self.beta, h0=self.h0)


def make_varlen_inputs(lengths, H: int, K: int, V: int, *, HV: int | None = None, per_k_gate: bool = False,
                       io_dtype: torch.dtype = torch.bfloat16, with_h0: bool = False,
                       seed: int = 0) -> VarlenInputs:
    """Draw a packed batch of len(lengths) sequences (see the module docstring)."""
    lengths = [int(x) for x in lengths]
    if not lengths or min(lengths) < 0:
        raise ValueError("lengths must be a non-empty list of non-negative integers")
    HV = H if HV is None else int(HV)
    total = sum(lengths)
    x = make_inputs(1, max(total, 1), HV, K, V, per_k_gate=per_k_gate, io_dtype=io_dtype, seed=seed)
    q, k, v, g, beta = (t[0, :total] for t in (x.q, x.k, x.v, x.g, x.beta))
    q, k = q[:, :H].contiguous(), k[:, :H].contiguous()
    h0 = None
    if with_h0:
        gen = torch.Generator(device="cpu")
        gen.manual_seed(seed + 1)
        h0 = 0.02 * torch.randn(len(lengths), HV, K, V, generator=gen, dtype=torch.float32)
    cu = torch.tensor([0] + lengths, dtype=torch.int64).cumsum(0).to(torch.int32)
    return VarlenInputs(q=q, k=k, v=v.contiguous(), g=g.contiguous(), beta=beta.contiguous(), h0=h0, cu=cu)


def make_workload_inputs(wl, seed: int = 0) -> GdrInputs:
    """Inputs for one named workload (a `workloads.Workload`)."""
    return make_inputs(wl.B, wl.T, wl.H, wl.K, wl.V, per_k_gate=wl.per_k_gate,
                       io_dtype=wl.torch_dtype, with_h0=wl.with_h0, seed=seed)
