"""gdr_forward_static_scratch: the forward for callers that cannot allocate
device memory themselves -- for example a plugin whose host framework owns all
device memory and hands out no side buffers, or a latency-critical loop that
must not call cudaMalloc.  Instead of a caller workspace it uses one fixed
scratch array inside the library, shared by every call on the device.

The checks, per case:
- a larger problem runs through the shared array first, so the array holds
  another problem's leftovers when the case's calls read it;
- then two calls in a row (two input seeds) through the shared array; each is
  bit-identical to gdr_forward with a caller workspace on the same variant (the
  kernels are deterministic, so any difference is a stale-scratch read), and
  each meets the workloads' bars against the float64 oracle;
- the cases cover both staged variants AUTO resolves to (the tensor-core stages
  for bf16 and fp16, the CUDA-core stages for fp32), both gates, C = 32 and 64,
  and the segment-parallel scan, whose maps and starts also live in the array.
A problem too large for the array is refused before anything runs.  This file
is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from chunked_gated_delta_prepare_gb300 import gdr
from chunked_gated_delta_prepare_gb300.inputs import make_inputs
from gpu_helpers import all_pairs, check_forward, dev, io_name

CASES = [  # (B, T, H, K, V, C, per-key-dim gate, io dtype, segments, variant AUTO runs)
    (1, 256, 2, 64, 64, 64, False, torch.float32, 0, "simt"),
    (2, 512, 4, 128, 128, 64, False, torch.bfloat16, 0, "tensor"),
    (1, 256, 2, 64, 128, 32, True, torch.bfloat16, 0, "tensor"),
    (1, 192, 2, 128, 64, 32, False, torch.bfloat16, 0, "tensor"),
    (1, 192, 2, 128, 128, 64, True, torch.bfloat16, 0, "tensor"),
    (1, 2048, 2, 64, 64, 64, False, torch.bfloat16, 4, "tensor"),
    (1, 192, 2, 64, 128, 32, True, torch.float16, 0, "tensor"),
    (2, 256, 2, 128, 128, 64, False, torch.float16, 0, "tensor"),
]

# run through the shared array before each case, so the case reads over another problem's leftovers
LARGER = (2, 1024, 4, 128, 128, 64, False, torch.bfloat16, 0)


def _run(x, C, segments, use_static):
    q, k, v, g, beta, h0 = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.h0))
    p = gdr.problem_for(q, v, g, C, None, "auto", segments)
    B, T, H, K = q.shape
    V = v.shape[-1]
    o = torch.full((B, T, H, V), float("nan"), device="cuda", dtype=q.dtype)
    hf = torch.full((B, H, K, V), float("nan"), device="cuda", dtype=torch.float32)
    if use_static:
        gdr.gdr_forward_static_scratch(p, q, k, v, g, beta, h0, o, hf)
    else:
        # the workspace forward on the variant the static call resolved to
        p.variant = gdr.VARIANTS[gdr.gdr_last_variant()]
        nbytes = gdr.gdr_forward_workspace_bytes(p)
        ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
        gdr.gdr_forward(p, q, k, v, g, beta, h0, o, hf, ws, nbytes)
    torch.cuda.synchronize()
    return o, hf, gdr.gdr_last_variant()


def _ids(c):
    return "x".join(map(str, c[:6])) + ("-kda" if c[6] else "-gdn") + "-" + io_name(c[7]) + (f"-S{c[8]}" if c[8] else "")


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_static_scratch_two_calls_match_workspace_forward_and_oracle(case):
    B, T, H, K, V, C, per_k, dtype, segments, expect = case
    LB, LT, LH, LK, LV, LC, lpk, ldt, lseg = LARGER
    big = make_inputs(LB, LT, LH, LK, LV, per_k_gate=lpk, io_dtype=ldt, with_h0=True, seed=30)
    _run(big, LC, lseg, use_static=True)                       # leaves its data in the shared array
    xs = [make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=dtype, with_h0=True, seed=s) for s in (31, 32)]
    got = []
    for x in xs:                                                # two calls in a row on the shared array
        o, hf, ran = _run(x, C, segments, use_static=True)
        assert ran == expect
        got.append((o.clone(), hf.clone()))
    assert gdr.gdr_get_device_status() == 0
    io = io_name(dtype)
    for x, (o, hf) in zip(xs, got):
        o_ref, hf_ref, ran = _run(x, C, segments, use_static=False)
        assert ran == expect
        assert torch.equal(o, o_ref) and torch.equal(hf, hf_ref), "static-scratch result differs from the workspace run"
        check_forward(x, o, hf, all_pairs(B, H), C, 1.0 / np.sqrt(K), io)
    assert gdr.gdr_get_device_status() == 0


def test_problem_larger_than_the_static_array_is_refused():
    lib = gdr.load()
    # 4 x 2048 tokens x 16 heads at K = V = 128, bf16: about 160 MiB of staged scratch
    p = gdr.make_problem(4, 2048, 16, 128, 128, 64, torch.bfloat16)
    p.variant = gdr.VARIANTS["tensor"]
    assert gdr.gdr_forward_workspace_bytes(p) > gdr.STATIC_SCRATCH_BYTES
    st = lib.gdr_forward_static_scratch(ctypes.byref(p), 16, 16, 16, 16, 16, None, 16, None, None)
    assert st == 5  # GDR_ERR_WORKSPACE, returned before anything is launched
    p.variant = gdr.VARIANTS["auto"]
    st = lib.gdr_forward_static_scratch(ctypes.byref(p), 16, 16, 16, 16, 16, None, 16, None, None)
    assert st == 5
    p_small = gdr.make_problem(1, 256, 2, 64, 64, 64, torch.float32)
    assert gdr.gdr_forward_workspace_bytes(p_small) <= gdr.STATIC_SCRATCH_BYTES


def test_fused_variant_is_not_offered():
    lib = gdr.load()
    p = gdr.make_problem(1, 256, 2, 64, 64, 64, torch.bfloat16)
    p.variant = gdr.VARIANTS["fused"]
    st = lib.gdr_forward_static_scratch(ctypes.byref(p), 16, 16, 16, 16, 16, None, 16, None, None)
    assert st == 8  # GDR_ERR_UNSUPPORTED
