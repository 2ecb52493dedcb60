"""gdr_forward_static_scratch: the forward for callers that cannot allocate
device memory themselves -- for example a plugin whose host framework owns all
device memory and hands out no side buffers, or a latency-critical loop that
must not call cudaMalloc.  Instead of a caller workspace it uses one fixed
scratch array inside the library, shared by every call on the device.

The checks: its results match gdr_forward (with a caller workspace) on two
calls in a row, so the second call is not disturbed by what the first left in
the shared array; and a problem too large for the array is refused before
anything runs.  This file is named to be collected last.
"""
import ctypes

import pytest
import torch

from chunked_gated_delta_prepare_gb300 import gdr
from chunked_gated_delta_prepare_gb300.inputs import make_inputs
from gpu_helpers import H_TOL, O_TOL, dev, io_name, max_abs, rel_frob

CASES = [  # (B, T, H, K, V, C, per-key-dim gate, io dtype)
    (1, 256, 2, 64, 64, 64, False, torch.float32),
    (2, 512, 4, 128, 128, 64, False, torch.bfloat16),
    (1, 256, 2, 64, 128, 32, True, torch.bfloat16),
]


def _run(x, C, use_static):
    q, k, v, g, beta, h0 = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.h0))
    p = gdr.problem_for(q, v, g, C)
    B, T, H, K = q.shape
    V = v.shape[-1]
    o = torch.full((B, T, H, V), float("nan"), device="cuda", dtype=q.dtype)
    hf = torch.full((B, H, K, V), float("nan"), device="cuda", dtype=torch.float32)
    if use_static:
        gdr.gdr_forward_static_scratch(p, q, k, v, g, beta, h0, o, hf)
    else:
        nbytes = gdr.gdr_forward_workspace_bytes(p)
        ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
        gdr.gdr_forward(p, q, k, v, g, beta, h0, o, hf, ws, nbytes)
    return o, hf


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])) + ("-kda" if c[6] else "-gdn")
                         + "-" + io_name(c[7]))
def test_static_scratch_matches_workspace_forward_on_two_calls(case):
    B, T, H, K, V, C, per_k, dtype = case
    xs = [make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=dtype, with_h0=True, seed=s) for s in (31, 32)]
    refs = [_run(x, C, use_static=False) for x in xs]
    torch.cuda.synchronize()
    got = [_run(x, C, use_static=True) for x in xs]      # two calls in a row on the shared array
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    io = io_name(dtype)
    for (o, hf), (o_ref, hf_ref) in zip(got, refs):
        assert max_abs(o, o_ref.double().cpu().numpy()) <= O_TOL[io]
        assert rel_frob(hf, hf_ref.double().cpu().numpy()) <= H_TOL[io]


def test_problem_larger_than_the_static_array_is_refused():
    lib = gdr.load()
    # 4 x 2048 tokens x 16 heads at K = V = 128, bf16: about 160 MiB of staged scratch
    p = gdr.make_problem(4, 2048, 16, 128, 128, 64, torch.bfloat16)
    assert gdr.gdr_forward_workspace_bytes(p) > gdr.STATIC_SCRATCH_BYTES
    st = lib.gdr_forward_static_scratch(ctypes.byref(p), 16, 16, 16, 16, 16, None, 16, None, None)
    assert st == 5  # GDR_ERR_WORKSPACE, returned before anything is launched
    p_small = gdr.make_problem(1, 256, 2, 64, 64, 64, torch.float32)
    assert gdr.gdr_forward_workspace_bytes(p_small) <= gdr.STATIC_SCRATCH_BYTES
