"""Throughput of the chunked gated-delta-rule forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
                    [--variant auto|simt|tensor|fused] [--seq-len T]

One step = one whole forward (gate cumsum, WY prepare, state scan, chunk output)
over one batch of the 32k-token GDN workload (B=1, T=32768, H=32, K=V=128, C=64,
bf16 io, fp32 state, h0 ~ N(0, 0.02)), inputs already resident in HBM.  Each
timed step is one gdr_forward call bracketed by CUDA events on the launching
stream; a 256 MiB buffer (about twice the L2) is overwritten before every timed
step, outside the events.  A separate pass calls the same kernels one by one
through their stage entry points to split the step by kernel.  Rank 0 prints
one JSON line.

The same line carries two more legs on the same workload: "backward" (the
gradient of o and h_final, stage by stage) and "varlen" (the workload's tokens
packed as eleven sequences of mixed length through gdr_varlen_forward).

--impl reference times the float64 CPU oracle (the only other implementation
of this computation) on the host cores, one bounded sample of the same workload
per step.

Under torchrun (N > 1) every rank runs its own copy of the workload on its own
GPU (the problem shards by (batch, head) with no exchange): weak scaling, and
`value` is the tokens all ranks processed divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from chunked_gated_delta_prepare_gb300 import gdr, workloads  # noqa: E402
from chunked_gated_delta_prepare_gb300.inputs import make_varlen_inputs, make_workload_inputs  # noqa: E402

METRIC = "gated-delta-rule fwd tokens/s at 1 GB300; achieved HBM GB/s & % roofline"
FLUSH_BYTES = 256 << 20


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# Algorithmic HBM bytes per (token, head) of each kernel, and per (batch, head)
# for the state.  e = io bytes, GW = 4 (scalar gate) or 4K (per-key-dim gate).
# with_p: the prepare also reads q and writes the gated scores P (C x C per
# chunk, so C e bytes per token), which the fused scan/output kernel reads.
def algorithmic_bytes(wl, kernel: str, with_p: bool = False, segs: int = 1) -> int:
    e = 2 if wl.io == "bf16" else 4
    K, V, C = wl.K, wl.V, wl.chunk
    gw = 4 * (K if wl.per_k_gate else 1)
    th = wl.B * wl.T * wl.H
    bh = wl.B * wl.H
    state = (4 * K * V if wl.with_h0 else 0) + 4 * K * V
    p_bytes = C * e if with_p else 0
    if kernel == "prepare":      # read k, v, g, beta (+ q); write w, u, g_cum (+ P)
        per = 2 * K * e + 2 * V * e + 2 * gw + e + (K * e + p_bytes if with_p else 0)
        return th * per
    if kernel == "scan":         # read k, w, u, g_cum; write v_new, checkpoint (K*V*e per chunk)
        per = 2 * K * e + 2 * V * e + gw + (K * V * e) // C
        return th * per + bh * state
    if kernel == "output":       # read q, k, v_new, g_cum, checkpoint; write o
        per = 2 * K * e + 2 * V * e + gw + (K * V * e) // C
        return th * per
    if kernel == "scan_output":  # read q, k, w, u, g_cum (+ P); write o; state in and out
        per = 3 * K * e + 2 * V * e + gw + p_bytes
        return th * per + bh * state
    if kernel == "gated_operands":   # per-key-dim gate: read q, k, g_cum; write P, qg, kg
        return th * (2 * K * e + gw + C * e + 2 * K * e)
    if kernel == "transfer":     # read k, w, u, g_cum; write each segment's M [K,K] and Z [K,V] (fp32)
        per = 2 * K * e + V * e + gw
        return th * per + segs * bh * 4 * (K * K + K * V)
    if kernel == "combine":      # read M, Z (and h0); write the segment starts and h_final (fp32)
        return segs * bh * 4 * (K * K + 2 * K * V) + bh * state
    if kernel == "forward":      # the I/O floor: read q, k, v, g, beta, h0; write o, h_final
        per = 2 * K * e + 2 * V * e + gw + e
        return th * per + bh * state
    raise ValueError(kernel)


def overlap_pieces(wl, variant: str, segments: int) -> int:
    """Pieces gdr_forward cuts one sequence into on the tcgen05 fused path (the library's rule: B = 1, no
    segments, at least 128 chunks; sizes from 16 chunks growing by 3/2, never below an equal share of what
    is left among at most 32 pieces); 1 when it does not."""
    NT = wl.NT
    if variant != "fused_tc" or segments != 1 or wl.B != 1 or NT < 128:
        return 1
    n = c = 0
    ln = 16
    while c < NT:
        ln = max(ln, -(-(NT - c) // (32 - n)))
        c = min(NT, c + ln)
        n += 1
        ln += ln // 2
    return n


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def traffic_for(kernel_name: str, workload: str):
    """DRAM bytes per launch of a kernel on a workload from the committed ncu summary, or
    None when there is no record or the kernel source changed after the counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            recs = json.load(f)["records"]
        rec = next(r for r in recs if r["kernel"] == kernel_name and r["workload"] == workload)
        src = os.path.join(ROOT, rec["source"])
        with open(src, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
        if digest != rec["source_sha256"]:
            return None
        return rec["bytes_per_launch"]
    except Exception:
        return None


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_throughput(world: int, tokens_per_rank_step: int, steps: int, slowest_seconds: float) -> float:
    """Tokens per second of the whole job: every rank runs its own full copy of the
    workload, so the job processed world x tokens x steps in the slowest rank's time."""
    return world * tokens_per_rank_step * steps / slowest_seconds


# ------------------------------------------------------------------ CPU oracle leg

def oracle_sample(wl, x, n_heads: int):
    """Time the float64 token-recurrence oracle on the first n_heads heads (all T tokens)."""
    import oracle
    pairs = [(b, h) for b in range(wl.B) for h in range(wl.H)][:n_heads]
    def tok(t):
        return torch.stack([t[b, :, h] for b, h in pairs]).unsqueeze(2)
    q, k, v, g, beta = (tok(t) for t in (x.q, x.k, x.v, x.g, x.beta))
    h0 = None if x.h0 is None else torch.stack([x.h0[b, h] for b, h in pairs]).unsqueeze(1)
    args = [oracle.chunked._f64(t) for t in (q, k, v, g, beta)] + [oracle.chunked._f64(h0)]
    cores = oracle.host_cores()
    t0 = time.perf_counter()
    oracle.naive_forward(*args, wl.chunk, 1.0 / wl.K ** 0.5, with_ckpt=False, nthreads=cores)
    dt = time.perf_counter() - t0
    token_heads = len(pairs) * wl.T
    return dict(seconds=dt, tokens_per_s=token_heads / wl.H / dt, cores=cores,
                sample=f"{len(pairs)} of {wl.B * wl.H} (batch, head) pairs x all {wl.T} tokens "
                       f"({token_heads} token-heads), float64 C token recurrence, {cores} threads")


def run_reference(args, wl):
    # rank 0 alone times the oracle; other ranks (under torchrun) exit without work
    if int(os.environ.get("RANK", "0")) != 0:
        return
    x = make_workload_inputs(wl)
    n_heads = max(1, min(wl.B * wl.H, args.ref_heads))
    for _ in range(args.warmup):
        oracle_sample(wl, x, n_heads)
    secs, last = 0.0, None
    for _ in range(args.steps):
        last = oracle_sample(wl, x, n_heads)
        secs += last["seconds"]
    tokens = n_heads * wl.T / wl.H * args.steps
    value = tokens / secs
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, the workload's distributions)",
            "config": dict(wl.describe(), sample=last["sample"]),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": last["cores"], "kind": "oracle",
                             "sample": last["sample"]},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU leg

def time_backward(args, wl, x, dev, flush, stream, world):
    """gdr_backward's launches on the same workload, called one by one through their
    C-ABI entry points (as gdr_backward calls them) so each can be timed; the upstream
    gradients do and dh_final are seeded normals."""
    B, T, H, K, V, C = wl.B, wl.T, wl.H, wl.K, wl.V, wl.chunk
    q, k, v, g, beta = (t.to(dev) for t in (x.q, x.k, x.v, x.g, x.beta))
    h0 = x.h0.to(dev) if x.h0 is not None else None
    gen = torch.Generator().manual_seed(7)
    d_o = torch.randn(B, T, H, V, generator=gen).to(q.dtype).to(dev)
    dhf = torch.randn(B, H, K, V, generator=gen).to(dev)
    p = gdr.problem_for(q, v, g, C, None, args.variant, args.segments)
    if gdr.gdr_backward_workspace_bytes(p) == 0:
        return None
    NT = -(-T // C)
    f32 = dict(device=dev, dtype=torch.float32)
    g_cum, w, u, v_new = torch.empty_like(g), torch.empty_like(k), torch.empty_like(v), torch.empty_like(v)
    h_ckpt = torch.empty(B, NT, H, K, V, device=dev, dtype=q.dtype)
    dv_loc, dv_new = torch.empty(B, T, H, V, **f32), torch.empty(B, T, H, V, **f32)
    dh_ckpt = torch.empty(B, NT, H, K, V, **f32)
    dk_part, dw = torch.empty(B, T, H, K, **f32), torch.empty(B, T, H, K, **f32)
    dG_part = torch.empty(g.shape, **f32)
    dq, dk, dv, dbeta = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(beta)
    dg, dh0 = torch.empty(g.shape, **f32), torch.empty(B, H, K, V, **f32)
    fast = q.dtype == torch.bfloat16 and g.dim() == 3 and args.variant in ("auto", "tensor")
    S = gdr.gdr_forward_segments(p) if q.dtype == torch.bfloat16 and args.variant != "simt" else 1
    launches_per_call = 1
    if S > 1:
        # segment-parallel: gdr_backward as one call (prepare, transfer, stitch, re-scan, [local term],
        # reverse scan twice around the reverse stitch, the per-chunk stage [+ its two filtered stages])
        nbytes = gdr.gdr_backward_workspace_bytes(p)
        ws = torch.empty(nbytes, device=dev, dtype=torch.uint8)
        hf0 = h0
        launches_per_call = 8 + (0 if fast and C == 64 else 1) + (0 if fast else 2)
        names = [f"backward_segmented_S{S}"]
        calls = [lambda: gdr.gdr_backward(p, q, k, v, g, beta, hf0, d_o, dhf, dq, dk, dv, dg, dbeta, dh0, ws, nbytes)]
    elif fast and C == 32:
        # the tensor-core path at 32-token chunks: the local term from its own kernel
        tinv = torch.empty(B, NT, H, C, C, device=dev, dtype=q.dtype)
        dv_loc16 = torch.empty(B, T, H, V, device=dev, dtype=q.dtype)
        dh_ckpt16 = torch.empty(B, NT, H, K, V, device=dev, dtype=q.dtype)
        dv_new16 = torch.empty(B, T, H, V, device=dev, dtype=q.dtype)
        names = ["prepare", "rescan", "dv_local", "scan_dh", "wy_dqkg"]
        calls = [lambda: gdr.gdr_bwd_prepare(p, q, k, v, g, beta, w, u, g_cum, None, tinv),
                 lambda: gdr.gdr_scan_h(p, k, w, u, g_cum, h0, h_ckpt, v_new, None),
                 lambda: gdr.gdr_bwd_dv_local_tc(p, q, k, g_cum, d_o, dv_loc16),
                 lambda: gdr.gdr_bwd_scan_dh_tc(p, q, k, w, g_cum, dv_loc16, d_o, dhf, dh_ckpt16, dv_new16, dh0),
                 lambda: gdr.gdr_bwd_wy_dqkg(p, q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o, dv_new16,
                                             dh_ckpt16, dq, dk, dv, dbeta, dg)]
    elif fast:
        # the tensor-core path gdr_backward takes here: four launches, bf16 intermediates
        P = torch.empty(B, NT, H, C, C, device=dev, dtype=q.dtype)
        tinv = torch.empty(B, NT, H, C, C, device=dev, dtype=q.dtype)
        dh_ckpt16 = torch.empty(B, NT, H, K, V, device=dev, dtype=q.dtype)
        dv_new16 = torch.empty(B, T, H, V, device=dev, dtype=q.dtype)
        names = ["prepare", "rescan", "scan_dh", "wy_dqkg"]
        calls = [lambda: gdr.gdr_bwd_prepare(p, q, k, v, g, beta, w, u, g_cum, P, tinv),
                 lambda: gdr.gdr_scan_h(p, k, w, u, g_cum, h0, h_ckpt, v_new, None),
                 lambda: gdr.gdr_bwd_scan_dh_p(p, q, k, w, g_cum, P, d_o, dhf, dh_ckpt16, dv_new16, dh0),
                 lambda: gdr.gdr_bwd_wy_dqkg(p, q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o, dv_new16,
                                             dh_ckpt16, dq, dk, dv, dbeta, dg)]
    elif q.dtype == torch.bfloat16 and args.variant in ("auto", "tensor"):
        # a per-key-dim gate: every stage on the tensor cores (bf16 intermediates); the CUDA-core
        # per-chunk stages run over the chunks the tensor-core one flags (with this workload's gate
        # none is, and their CTAs return at once)
        tinv = torch.empty(B, NT, H, C, C, device=dev, dtype=q.dtype)
        flags = torch.empty(B, NT, H, device=dev, dtype=torch.int32)
        dv_loc16 = torch.empty(B, T, H, V, device=dev, dtype=q.dtype)
        dh_ckpt16 = torch.empty(B, NT, H, K, V, device=dev, dtype=q.dtype)
        dv_new16 = torch.empty(B, T, H, V, device=dev, dtype=q.dtype)
        names = ["prepare", "rescan", "dv_local", "scan_dh", "wy_dqkg", "dqkwg_flagged", "wy_flagged"]
        calls = [lambda: gdr.gdr_bwd_prepare(p, q, k, v, g, beta, w, u, g_cum, None, tinv),
                 lambda: gdr.gdr_scan_h(p, k, w, u, g_cum, h0, h_ckpt, v_new, None),
                 lambda: gdr.gdr_bwd_dv_local_tc(p, q, k, g_cum, d_o, dv_loc16),
                 lambda: gdr.gdr_bwd_scan_dh_tc(p, q, k, w, g_cum, dv_loc16, d_o, dhf, dh_ckpt16, dv_new16, dh0),
                 lambda: gdr.gdr_bwd_wy_dqkg(p, q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o, dv_new16,
                                             dh_ckpt16, dq, dk, dv, dbeta, dg, flags),
                 lambda: gdr.gdr_bwd_dqkwg(p, q, k, v_new, g_cum, h_ckpt, dh_ckpt16, d_o, dv_new16, dq, dk_part, dw,
                                           dG_part, flags),
                 lambda: gdr.gdr_bwd_wy(p, k, v, beta, g_cum, dw, dv_new16, dk_part, dG_part, dk, dv, dbeta, dg,
                                        flags)]
    else:
        names = ["prepare", "rescan", "dv_local", "scan_dh", "dqkwg", "wy"]
        calls = [lambda: gdr.gdr_prepare_wy(p, k, v, g, beta, w, u, g_cum),
                 lambda: gdr.gdr_scan_h(p, k, w, u, g_cum, h0, h_ckpt, v_new, None),
                 lambda: gdr.gdr_bwd_dv_local(p, q, k, g_cum, d_o, dv_loc),
                 lambda: gdr.gdr_bwd_scan_dh(p, q, k, w, g_cum, d_o, dv_loc, dhf, dh_ckpt, dv_new, dh0),
                 lambda: gdr.gdr_bwd_dqkwg(p, q, k, v_new, g_cum, h_ckpt, dh_ckpt, d_o, dv_new, dq, dk_part, dw,
                                           dG_part),
                 lambda: gdr.gdr_bwd_wy(p, k, v, beta, g_cum, dw, dv_new, dk_part, dG_part, dk, dv, dbeta, dg)]
    ran = []
    for f in calls:
        f()
        ran.append(gdr.gdr_last_variant())
    steps = max(3, min(args.steps, 10))
    for _ in range(args.warmup):
        flush.fill_(1)
        for f in calls:
            f()
    torch.cuda.synchronize()
    n = len(calls)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for s in range(steps):
        flush.fill_(s & 0xFF)
        evs[s][0].record(stream)
        for i, f in enumerate(calls):
            f()
            evs[s][i + 1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    if gdr.gdr_get_device_status() != 0:
        raise RuntimeError("device status set after the backward's timed region")
    per = [sum(evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(steps)) / steps for i in range(n)]
    total_s = max_over_ranks(sum(evs[s][0].elapsed_time(evs[s][n]) for s in range(steps)) / 1e3, world)
    return {"ms_per_step": 1e3 * total_s / steps, "steps": steps,
            "value": weak_scaling_throughput(world, B * T, steps, total_s), "unit": "tokens/s",
            "kernel_ms": {f"{names[i]}[{ran[i]}]": per[i] for i in range(n)},
            "gpu_launches": n * launches_per_call * steps, "segments": S,
            "upstream": "do ~ N(0,1) in the io dtype, dh_final ~ N(0,1) fp32, seed 7"}


# packed variable-length leg: the workload's tokens as eleven sequences of mixed length (one empty,
# one a single token, ragged tails), the mix given here for 32768 tokens and scaled to other totals
VARLEN_MIX = [8192, 4096, 4133, 1, 6000, 0, 2048, 3000, 777, 2911, 1610]


def varlen_lengths(total: int):
    out = [n * total // sum(VARLEN_MIX) for n in VARLEN_MIX]
    out[0] += total - sum(out)
    return out


def time_varlen(args, wl, dev, flush, stream, world):
    """gdr_varlen_forward on the workload's B T tokens packed as VARLEN_MIX: one C-ABI call per step.
    On the fused path at 64-token chunks it runs chunk-packed with the packed tensors read and o written in
    place (the chunk map, the prepare, the fused scan and output walking each sequence's chunks); on the
    other tensor-core paths chunk-packed through copies (the pack, the prepare, the scan and output, the
    unpack); on the CUDA cores padded (the pack, gdr_forward on rows as long as the longest sequence, the
    unpack)."""
    lengths = varlen_lengths(wl.B * wl.T)
    x = make_varlen_inputs(lengths, wl.H, wl.K, wl.V, per_k_gate=wl.per_k_gate, io_dtype=wl.torch_dtype,
                           with_h0=wl.with_h0, seed=0)
    q, k, v, g, beta = (t.to(dev) for t in (x.q, x.k, x.v, x.g, x.beta))
    h0 = x.h0.to(dev) if x.h0 is not None else None
    cu_dev = x.cu.to(dev)
    total = int(x.cu[-1])
    p = gdr.varlen_problem(q, v, g, x.cu, None, wl.chunk, None, args.variant, args.segments)
    o = torch.empty_like(v)
    hf = torch.empty(int(p.B), wl.H, wl.K, wl.V, device=dev, dtype=torch.float32)
    nbytes = gdr.gdr_varlen_forward_workspace_bytes(p)
    ws = torch.empty(nbytes, device=dev, dtype=torch.uint8)

    def call():
        gdr.gdr_varlen_forward(p, x.cu, cu_dev, total, q, k, v, g, beta, h0, o, hf, ws, nbytes)

    call()
    variant = gdr.gdr_last_variant()
    C = wl.chunk
    chunked = variant != "simt" and total > 0
    S = 1 if chunked else gdr.gdr_forward_segments(p)
    if chunked and variant == "fused" and C == 64:   # q, k, v, g, beta read and o written in place
        layout, working = "chunk-packed, read in place", sum(-(-n // C) * C for n in lengths)
        launches = 3
    elif chunked:
        layout, working = "chunk-packed", sum(-(-n // C) * C for n in lengths)
        launches = 3 + (2 if variant == "fused" else 3)
    else:
        layout, working = "padded", int(p.B * p.T)
        launches = 2 + (2 if variant == "fused" else 3) + (2 if S > 1 else 0)
    steps = max(3, min(args.steps, 10))
    for _ in range(args.warmup):
        flush.fill_(1)
        call()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for s in range(steps):
        flush.fill_(s & 0xFF)
        evs[s][0].record(stream)
        call()
        evs[s][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    if gdr.gdr_get_device_status() != 0:
        raise RuntimeError("device status set after the packed forward's timed region")
    total_s = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / 1e3, world)

    # the backward of the same packed batch: gdr_varlen_backward, one call per step
    gen = torch.Generator().manual_seed(7)
    d_o = torch.randn(v.shape, generator=gen).to(v.dtype).to(dev)
    dhf = torch.randn(hf.shape, generator=gen).to(dev)
    grads = [torch.empty_like(t) for t in (q, k, v, g, beta)]
    dh0 = torch.empty_like(hf)
    bbytes = gdr.gdr_varlen_backward_workspace_bytes(p)
    bws = torch.empty(bbytes, device=dev, dtype=torch.uint8)

    def bcall():
        gdr.gdr_varlen_backward(p, x.cu, cu_dev, total, q, k, v, g, beta, h0, d_o, dhf, *grads, dh0, bws, bbytes)

    bcall()
    bvariant = gdr.gdr_last_variant()
    for _ in range(args.warmup):
        flush.fill_(1)
        bcall()
    torch.cuda.synchronize()
    bevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for s in range(steps):
        flush.fill_(s & 0xFF)
        bevs[s][0].record(stream)
        bcall()
        bevs[s][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    if gdr.gdr_get_device_status() != 0:
        raise RuntimeError("device status set after the packed backward's timed region")
    bwd_s = max_over_ranks(sum(a.elapsed_time(b) for a, b in bevs) / 1e3, world)
    return {"ms_per_step": 1e3 * total_s / steps, "steps": steps,
            "value": weak_scaling_throughput(world, total, steps, total_s), "unit": "tokens/s",
            "backward": {"ms_per_step": 1e3 * bwd_s / steps, "variant": bvariant,
                         "value": weak_scaling_throughput(world, total, steps, bwd_s), "unit": "tokens/s"},
            "sequences": len(lengths), "lengths": lengths, "layout": layout, "working_tokens": working,
            "variant": variant, "segments": S,
            "gpu_launches": launches * steps}


def run_ours(args, wl):
    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    x = make_workload_inputs(wl)
    q, k, v, g, beta = (t.to(dev) for t in (x.q, x.k, x.v, x.g, x.beta))
    h0 = x.h0.to(dev) if x.h0 is not None else None
    B, T, H, K, V, C = wl.B, wl.T, wl.H, wl.K, wl.V, wl.chunk
    p = gdr.problem_for(q, v, g, C, None, args.variant, args.segments)
    S = gdr.gdr_forward_segments(p)
    o = torch.empty(B, T, H, V, device=dev, dtype=q.dtype)
    hf = torch.empty(B, H, K, V, device=dev, dtype=torch.float32)
    nbytes = gdr.gdr_forward_workspace_bytes(p)
    ws = torch.empty(max(nbytes, 1), device=dev, dtype=torch.uint8)
    flush = torch.empty(FLUSH_BYTES, device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream()

    # Probe which variant gdr_forward runs, and how its work splits into launches.
    gdr.gdr_forward(p, q, k, v, g, beta, h0, o, hf, ws if nbytes else None, nbytes)
    torch.cuda.synchronize()
    variant = gdr.gdr_last_variant()
    fused = variant in ("fused", "fused_tc")
    staged = not fused
    P = None
    # the segment-parallel scan (S > 1): every segment's map, the stitch, then the scan of all
    # segments at once on the view of B S sequences of T / S tokens
    seg_calls, seg_names, vp = [], [], None
    if S > 1:
        Hk = q.shape[2]
        M = torch.empty(B, S, H, K, K, device=dev)
        Z = torch.empty(B, S, H, K, V, device=dev)
        starts = torch.empty(B, S, H, K, V, device=dev)
        vp = gdr.problem_for(q, v, g, C, None, args.variant, 1)
        vp.B, vp.T = B * S, T // S
        seg_names = ["transfer", "combine"]
        seg_calls = [lambda: gdr.gdr_scan_transfer(sp, k, w, u, g_cum, S, M, Z),
                     lambda: gdr.gdr_scan_combine(sp, S, M, Z, h0, starts, hf)]
        del Hk
    if fused and wl.per_k_gate:
        # the per-key-dim gate on the tcgen05 path: the prepare, the gated operands P, qg, kg, then the scan
        # and output on them
        g_cum = torch.empty_like(g)
        w = torch.empty_like(k)
        u = torch.empty_like(v)
        P = torch.empty(B, -(-T // C), H, C, C, device=dev, dtype=q.dtype)
        qg = torch.empty(B, T, H, K, device=dev, dtype=q.dtype)
        kg = torch.empty(B, T, H, K, device=dev, dtype=q.dtype)
        sp = gdr.problem_for(q, v, g, C, None, "fused_tc", 1)   # the stage call takes the gated operands there
        if vp is not None:
            vp.variant = gdr.VARIANTS["fused_tc"]
        kernels = ["prepare", "gated_operands"] + seg_names + ["scan_output"]

        def launches():
            scan = (lambda: gdr.gdr_scan_output(vp, qg, kg, w, u, g_cum, P, starts, o, None)) if vp is not None else \
                (lambda: gdr.gdr_scan_output(sp, qg, kg, w, u, g_cum, P, h0, o, hf))
            return [lambda: gdr.gdr_prepare_wy(sp, k, v, g, beta, w, u, g_cum),
                    lambda: gdr.gdr_gated_operands(sp, q, k, g_cum, P, kg, qg)] + seg_calls + [scan]
    elif fused:
        # the two kernels gdr_forward runs on this path, called one by one so each can be timed
        g_cum = torch.empty_like(g)
        w = torch.empty_like(k)
        u = torch.empty_like(v)
        P = torch.empty(B, -(-T // C), H, C, C, device=dev, dtype=q.dtype) if C == 64 and args.p_from == "prepare" else None
        sp = gdr.problem_for(q, v, g, C, None, args.variant, 1)
        kernels = ["prepare"] + seg_names + ["scan_output"]

        def launches():
            prep = (lambda: gdr.gdr_prepare_wy(sp, k, v, g, beta, w, u, g_cum)) if P is None else \
                (lambda: gdr.gdr_prepare_wyp(sp, q, k, v, g, beta, w, u, g_cum, P))
            if vp is not None:
                return [prep] + seg_calls + [lambda: gdr.gdr_scan_output(vp, q, k, w, u, g_cum, P, starts, o, None)]
            return [prep, lambda: gdr.gdr_scan_output(sp, q, k, w, u, g_cum, P, h0, o, hf)]
    elif staged:
        NT = -(-T // C)
        e = q.element_size()
        # the same three kernels gdr_forward runs, called one by one so each can be timed
        g_cum = torch.empty_like(g)
        w = torch.empty_like(k)
        u = torch.empty_like(v)
        v_new = torch.empty_like(v)
        h_ckpt = torch.empty(B, NT, H, K, V, device=dev, dtype=q.dtype)
        sp = gdr.problem_for(q, v, g, C, None, args.variant, 1)
        kernels = ["prepare"] + seg_names + ["scan", "output"]

        def launches():
            if vp is not None:
                scan = lambda: gdr.gdr_scan_h(vp, k, w, u, g_cum, starts, h_ckpt, v_new, None)
            else:
                scan = lambda: gdr.gdr_scan_h(sp, k, w, u, g_cum, h0, h_ckpt, v_new, hf)
            return [lambda: gdr.gdr_prepare_wy(sp, k, v, g, beta, w, u, g_cum)] + seg_calls + \
                [scan, lambda: gdr.gdr_chunk_output(sp, q, k, v_new, h_ckpt, g_cum, o)]
        del e

    # The headline: one gdr_forward call per step, events on the launching stream around it.
    def forward_call():
        gdr.gdr_forward(p, q, k, v, g, beta, h0, o, hf, ws if nbytes else None, nbytes)

    for _ in range(args.warmup):
        flush.fill_(1)
        forward_call()
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for s in range(args.steps):
            flush.fill_(s & 0xFF)
            evs[s][0].record(stream)
            forward_call()
            evs[s][1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    status = gdr.gdr_get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_s = max_over_ranks(sum(step_ms) / 1e3, world)
    value = weak_scaling_throughput(world, B * T, args.steps, total_s)

    # The split: the same kernels gdr_forward launches, called one by one through their stage entry
    # points in a separate timed pass, so each kernel's share of the step can be read.
    calls = launches()
    stage_variant = []
    for f in calls:
        f()
        stage_variant.append(gdr.gdr_last_variant())
    for _ in range(args.warmup):
        flush.fill_(1)
        for f in calls:
            f()
    torch.cuda.synchronize()
    assert gdr.gdr_get_device_status() == 0
    n = len(calls)
    split_steps = max(3, min(args.steps, 10))
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(split_steps)]
    torch.cuda.synchronize()
    for s in range(split_steps):
        flush.fill_(s & 0xFF)
        sevs[s][0].record(stream)
        for i, f in enumerate(calls):
            f()
            sevs[s][i + 1].record(stream)
    torch.cuda.synchronize()
    if gdr.gdr_get_device_status() != 0:
        raise RuntimeError("device status set after the split pass")
    avg_ms = [sum(sevs[s][i].elapsed_time(sevs[s][i + 1]) for s in range(split_steps)) / split_steps
              for i in range(n)]
    split_step_ms = sum(sevs[s][0].elapsed_time(sevs[s][n]) for s in range(split_steps)) / split_steps

    pieces = overlap_pieces(wl, variant, S)

    # Roofline of the dominant kernel.  "achieved" counts the forward's algorithmic bytes (the I/O
    # floor: q, k, v, g, beta read once, o written once, the state in and out) over that kernel's
    # average launch time; "frac_own_io" counts instead the bytes that kernel itself must move in this
    # kernel split (its inputs and outputs, intermediates included).
    hbm_gbs, _, peak_kind = peaks()
    dom = max(range(n), key=lambda i: avg_ms[i])
    dom_name = kernels[dom]
    floor_bytes = algorithmic_bytes(wl, "forward")
    own_bytes = algorithmic_bytes(wl, dom_name, with_p=fused and P is not None, segs=S)
    achieved = floor_bytes / (avg_ms[dom] / 1e3) / 1e9
    kname = {"prepare": "prepare_mma_kernel", "scan": "scan_mma_kernel", "output": "tc_output_kernel",
             "scan_output": "tc_scan_output_kernel" if variant == "fused_tc" else "fused_scan_output_kernel",
             "transfer": "scan_mma_kernel<transfer>", "combine": "segment_combine_kernel",
             "gated_operands": "tc_output_kernel<gated operands>"}[dom_name]
    if stage_variant[dom] == "simt":
        kname = f"simt_{dom_name}_kernel"
    traffic = traffic_for(kname, wl.name)

    # end to end through the public API: pinned host inputs in, o and h_final back to host
    hx = {n_: t.pin_memory() for n_, t in x.tensors().items() if t is not None}
    h2d = sum(t.numel() * t.element_size() for t in hx.values())
    d2h = o.numel() * o.element_size() + hf.numel() * hf.element_size()
    o_host = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)     # the caller's result buffers, pinned once
    hf_host = torch.empty(hf.shape, dtype=hf.dtype, pin_memory=True)
    for _ in range(2):
        gdr.forward(hx["q"], hx["k"], hx["v"], hx["g"], hx["beta"], hx.get("h0"), chunk=C, variant=args.variant,
                    workspace=ws, segments=args.segments, out=o_host, h_final_out=hf_host)
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 10))
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        oo, hh = gdr.forward(hx["q"], hx["k"], hx["v"], hx["g"], hx["beta"], hx.get("h0"), chunk=C,
                             variant=args.variant, workspace=ws, segments=args.segments, out=o_host,
                             h_final_out=hf_host)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_value = weak_scaling_throughput(world, B * T, e2e_steps, e2e_s)

    bwd = None if args.no_backward else time_backward(args, wl, x, dev, flush, stream, world)
    vl = None if args.no_varlen else time_varlen(args, wl, dev, flush, stream, world)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = oracle_sample(wl, x, max(1, min(wl.B * wl.H, args.cpu_heads)))

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.io == "bf16" else "f32",
            "data": "synthetic (seeded; q,k unit-norm, v N(0,1), beta sigmoid, g logsigmoid/16)",
            "config": dict(wl.describe(), variant=variant, l2="256 MiB buffer overwritten before every timed step",
                           kernels_per_step=2 * pieces if pieces > 1 else n, segments=S, pieces=pieces),
            "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "peak_source": f"{peak_kind} HBM copy bandwidth",
                         "traffic": traffic, "algorithmic_bytes_per_launch": floor_bytes,
                         "algorithmic_bytes": "the forward's I/O floor (q, k, v, g, beta, h0 in; o, h_final out)",
                         "avg_launch_ms": avg_ms[dom],
                         "frac_own_io": own_bytes / (avg_ms[dom] / 1e3) / 1e9 / hbm_gbs,
                         "own_io_bytes_per_launch": own_bytes},
            "kernel_ms": {f"{kernels[i]}[{stage_variant[i]}]": avg_ms[i] for i in range(n)},
            "split_ms_per_step": split_step_ms,
            "floor_roofline_frac": (floor_bytes / (hbm_gbs * 1e9)) / (total_s / args.steps),
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": (2 * pieces if pieces > 1 else n) * args.steps,
            "timed": "events around one gdr_forward call per step; kernel_ms from a separate pass of its stage calls",
            "clocks": clk.summary(),
        }
        if bwd is not None:
            line["backward"] = bwd
        if vl is not None:
            line["varlen"] = vl
        if cpu is not None:
            line["cpu_baseline"] = {"value": cpu["tokens_per_s"], "unit": "tokens/s", "cores": cpu["cores"],
                                    "kind": "oracle", "sample": cpu["sample"]}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=workloads.THROUGHPUT.name, choices=sorted(workloads.BY_NAME))
    ap.add_argument("--variant", default="auto", choices=sorted(gdr.VARIANTS))
    ap.add_argument("--segments", type=int, default=0,
                    help="segment-parallel scan: 0 = the library's choice, 1 = serial, S = S segments")
    ap.add_argument("--cpu-heads", type=int, default=32, help="heads in the CPU-oracle baseline sample")
    ap.add_argument("--ref-heads", type=int, default=4, help="heads per step of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true", help="skip timing the backward pass")
    ap.add_argument("--no-varlen", action="store_true", help="skip timing the packed variable-length forward")
    ap.add_argument("--p-from", choices=["prepare", "scan"], default="prepare",
                    help="fused path: gated scores P written by the prepare, or formed inside the scan kernel")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="run the workload at another T (small profiling captures only; not a bench line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    wl = workloads.BY_NAME[args.workload]
    if args.seq_len is not None:
        wl = wl.with_tokens(args.seq_len)
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
