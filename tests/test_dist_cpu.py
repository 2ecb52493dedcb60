"""The benchmark's multi-process path on CPU: two gloo ranks on this host.

Each rank of a multi-GPU run works on its own copy of the workload (the
(batch, head) problems are independent, so no data moves between ranks); the
ranks meet only at the barriers around the timed region and in one max-reduce of
the elapsed time.  These tests run that host logic with world size 2.
"""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))


def _rank_timing(rank, world, port, out):
    _env(rank, world, port)
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank reports its own elapsed seconds; the job is as slow as the slowest
    slowest = bench.max_over_ranks(1.0 + rank, w)
    out[rank] = (slowest, bench.weak_scaling_throughput(w, 1000, 4, slowest))
    bench.barrier(w)
    dist.destroy_process_group()


def _rank_reference(rank, world, port, out):
    _env(rank, world, port)
    sys.path.insert(0, ROOT)
    import contextlib
    import io
    import bench
    from chunked_gated_delta_prepare_gb300 import workloads
    buf = io.StringIO()
    args = type("A", (), dict(warmup=0, steps=1, ref_heads=1, gpus=world))()
    with contextlib.redirect_stdout(buf):
        if rank != 0:
            bench.run_reference(args, workloads.GDN_F32_T256)
    out[rank] = buf.getvalue()


def _spawn(fn, world=2):
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=fn, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        return codes, dict(out)


def test_two_gloo_ranks_agree_on_the_slowest_time():
    codes, out = _spawn(_rank_timing)
    assert codes == [0, 0]
    for r in (0, 1):
        slowest, value = out[r]
        assert slowest == 2.0
        # 2 ranks x 1000 tokens x 4 steps in 2 s
        assert value == pytest.approx(4000.0)


def test_reference_arm_idles_on_other_ranks():
    codes, out = _spawn(_rank_reference)
    assert codes == [0, 0]
    assert out[1] == ""


def test_weak_scaling_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.weak_scaling_throughput(1, 32768, 10, 0.02)
    two = bench.weak_scaling_throughput(2, 32768, 10, 0.02)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(32768 * 10 / 0.02)


def test_seq_len_override_keeps_the_problem_shape():
    from chunked_gated_delta_prepare_gb300 import workloads
    wl = workloads.THROUGHPUT.with_tokens(4096)
    assert (wl.B, wl.T, wl.H, wl.K, wl.V, wl.chunk) == (1, 4096, 32, 128, 128, 64)
    assert wl.name == "gdn_bf16_b1_t4096_h32_d128_c64"
    wl = workloads.THROUGHPUT.with_tokens(100)          # a partial last chunk is a valid problem
    assert (wl.T, wl.NT) == (100, 2)
    with pytest.raises(ValueError):
        workloads.THROUGHPUT.with_tokens(0)


def test_varlen_mix_covers_every_token():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.varlen_lengths(32768) == bench.VARLEN_MIX
    for total in (1, 100, 4096, 16384, 65536, 100003):
        lengths = bench.varlen_lengths(total)
        assert sum(lengths) == total and min(lengths) >= 0 and len(lengths) == len(bench.VARLEN_MIX)


def test_varlen_problem_from_packed_tensors():
    # the padded problem of a packed batch: B = sequences, T = the longest one (or the caller's row length)
    import torch
    from chunked_gated_delta_prepare_gb300 import gdr
    from chunked_gated_delta_prepare_gb300.inputs import make_varlen_inputs
    x = make_varlen_inputs([5, 0, 70, 12], 1, 64, 128, HV=2, per_k_gate=True, io_dtype=torch.bfloat16)
    assert x.cu.tolist() == [0, 5, 5, 75, 87]
    p = gdr.varlen_problem(x.q, x.v, x.g, x.cu, None, 64, None, "auto", 0)
    assert (p.B, p.T, p.H, p.K, p.V, p.chunk, p.HV, p.gate, p.io_dtype) == (4, 70, 1, 64, 128, 64, 2, 1, 1)
    p = gdr.varlen_problem(x.q, x.v, x.g, x.cu, 128, 64, None, "auto", 0)
    assert p.T == 128
    e = make_varlen_inputs([0, 0], 2, 64, 64)
    assert gdr.varlen_problem(e.q, e.v, e.g, e.cu, None, 64, None, "auto", 0).T == 1   # no tokens: rows of one
    with pytest.raises(ValueError):
        gdr.varlen_problem(e.q, e.v, e.g, torch.tensor([0], dtype=torch.int32), None, 64, None, "auto", 0)


def test_host_cu_accepts_lists_and_tensors():
    import torch
    from chunked_gated_delta_prepare_gb300 import gdr
    for cu in ([0, 3, 3, 10], torch.tensor([0, 3, 3, 10]), torch.tensor([0, 3, 3, 10], dtype=torch.int32)):
        h = gdr._host_cu(cu)
        assert h.dtype == torch.int32 and h.device.type == "cpu" and h.is_contiguous()
        assert h.tolist() == [0, 3, 3, 10]
