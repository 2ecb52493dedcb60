"""The C ABI under CUDA graph capture: gdr_forward, gdr_backward and
gdr_varlen_forward (with a device cu_seqlens) captured once into a
torch.cuda.CUDAGraph and replayed on new inputs copied into the captured
buffers.  Nothing in these calls synchronises, allocates or copies from pageable
memory, so capture records every launch.  The forward kernels are deterministic,
so a replay equals an eager call on the same inputs bit for bit; the backward's
row sums use atomics, so its replay is held to the parity bar instead.
"""
import pytest
import torch

from chunked_gated_delta_prepare_gb300 import gdr
from chunked_gated_delta_prepare_gb300.inputs import make_inputs, make_varlen_inputs
from gpu_helpers import dev, scaled_err

pytestmark = pytest.mark.gpu


def _fill(static, fresh):
    for s, f in zip(static, fresh):
        if s is not None:
            s.copy_(f)


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # warm-up off the capture, as torch's graph recipe asks
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


@pytest.mark.parametrize("variant,dtype,per_k,B,T", [("fused", torch.bfloat16, False, 2, 320),
                                                     ("fused_tc", torch.bfloat16, False, 2, 320),
                                                     ("fused_tc", torch.bfloat16, False, 1, 64 * 64 * 2 + 50),
                                                     ("tensor", torch.bfloat16, True, 2, 320),
                                                     ("simt", torch.float32, False, 2, 320)])
def test_forward_replays_in_a_graph(variant, dtype, per_k, B, T):
    # (the single long sequence on fused_tc runs overlapped: its internal stream forks from and joins the
    # captured stream)
    H, C = 3, 64
    K, V = 128, 128 if variant == "fused_tc" else 64
    xs = [make_inputs(B, T, H, K, V, per_k_gate=per_k, io_dtype=dtype, with_h0=True, seed=s) for s in (0, 1)]
    q, k, v, g, beta, h0 = (dev(t) for t in xs[0].tensors().values())
    p = gdr.problem_for(q, v, g, C, None, variant)
    o = torch.empty(B, T, H, V, device="cuda", dtype=dtype)
    hf = torch.empty(B, H, K, V, device="cuda")
    nbytes = gdr.gdr_forward_workspace_bytes(p)
    ws = torch.empty(max(nbytes, 1), device="cuda", dtype=torch.uint8)
    graph = _capture(lambda: gdr.gdr_forward(p, q, k, v, g, beta, h0, o, hf, ws, nbytes))
    for x in xs:
        _fill((q, k, v, g, beta, h0), x.tensors().values())
        graph.replay()
        torch.cuda.synchronize()
        o_g, hf_g = o.clone(), hf.clone()
        gdr.gdr_forward(p, q, k, v, g, beta, h0, o, hf, ws, nbytes)
        torch.cuda.synchronize()
        assert gdr.gdr_get_device_status() == 0
        assert torch.equal(o_g, o) and torch.equal(hf_g, hf)


def test_backward_replays_in_a_graph():
    B, T, H, K, V, C = 1, 384, 2, 128, 128, 64
    xs = [make_inputs(B, T, H, K, V, io_dtype=torch.bfloat16, with_h0=True, seed=s) for s in (2, 3)]
    gen = torch.Generator().manual_seed(4)
    ups = [(torch.randn(B, T, H, V, generator=gen).to(torch.bfloat16), torch.randn(B, H, K, V, generator=gen))
           for _ in xs]
    q, k, v, g, beta, h0 = (dev(t) for t in xs[0].tensors().values())
    d_o, dhf = dev(ups[0][0]), dev(ups[0][1])
    p = gdr.problem_for(q, v, g, C)
    outs = [torch.empty_like(t) for t in (q, k, v, g, beta)] + [torch.empty(B, H, K, V, device="cuda")]
    nbytes = gdr.gdr_backward_workspace_bytes(p)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)

    def run():
        gdr.gdr_backward(p, q, k, v, g, beta, h0, d_o, dhf, *outs, ws, nbytes)

    graph = _capture(run)
    for x, (do_, dhf_) in zip(xs, ups):
        _fill((q, k, v, g, beta, h0, d_o, dhf), list(x.tensors().values()) + [do_, dhf_])
        graph.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in outs]
        run()
        torch.cuda.synchronize()
        assert gdr.gdr_get_device_status() == 0
        for a, b in zip(got, outs):
            assert scaled_err(a, b.double().cpu().numpy()) <= 1e-2


def test_varlen_forward_replays_in_a_graph():
    lengths = [100, 0, 1, 64, 200]
    xs = [make_varlen_inputs(lengths, 2, 128, 128, io_dtype=torch.bfloat16, with_h0=True, seed=s) for s in (5, 6)]
    q, k, v, g, beta, h0 = (dev(t) for t in xs[0].tensors().values())
    cu_host, cu_dev = xs[0].cu, xs[0].cu.to("cuda")
    p = gdr.varlen_problem(q, v, g, cu_host, None, 64, None, "auto", 0)
    total = int(cu_host[-1])
    o = torch.empty_like(v)
    hf = torch.empty(len(lengths), 2, 128, 128, device="cuda")
    nbytes = gdr.gdr_varlen_forward_workspace_bytes(p)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8)

    def run():
        gdr.gdr_varlen_forward(p, cu_host, cu_dev, total, q, k, v, g, beta, h0, o, hf, ws, nbytes)

    graph = _capture(run)
    for x in xs:
        _fill((q, k, v, g, beta, h0), x.tensors().values())
        graph.replay()
        torch.cuda.synchronize()
        o_g, hf_g = o.clone(), hf.clone()
        run()
        torch.cuda.synchronize()
        assert gdr.gdr_get_device_status() == 0
        assert torch.equal(o_g, o) and torch.equal(hf_g, hf)
