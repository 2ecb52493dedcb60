"""ctypes binding of libgdr (include/gdr.h).

Argument marshalling only: every step of the forward runs in libgdr's CUDA
kernels.  PyTorch supplies device memory and the current stream.  There is no
CPU fallback: if the library is missing or cannot load, every call raises.

The functions mirror the C ABI names:
    gdr_prepare_wy, gdr_prepare_wyp, gdr_scan_h, gdr_scan_transfer, gdr_scan_combine, gdr_scan_combine_reverse,
    gdr_chunk_output,
    gdr_scan_output, gdr_forward, gdr_forward_workspace_bytes, gdr_forward_segments, gdr_bwd_dv_local, gdr_bwd_scan_dh, gdr_bwd_dqkwg, gdr_bwd_wy,
    gdr_bwd_prepare, gdr_bwd_scan_dh_p, gdr_bwd_wy_dqkg, gdr_backward, gdr_backward_workspace_bytes,
    gdr_varlen_forward, gdr_varlen_forward_workspace_bytes, gdr_varlen_backward,
    gdr_varlen_backward_workspace_bytes,
    gdr_status_string, gdr_get_device_status, gdr_selftest_bounded_wait,
    gdr_last_variant, gdr_version
and `forward(...)` / `backward(...)` are the convenience calls that allocate outputs and
the workspace (and, given CPU tensors, copy them to the GPU and the results back);
`forward_varlen(...)` / `backward_varlen(...)` the same for packed variable-length sequences.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libgdr.so")

GDR_OK = 0
STATUS_NAMES = {0: "GDR_OK", 1: "GDR_ERR_NULL", 2: "GDR_ERR_SHAPE", 3: "GDR_ERR_DTYPE", 4: "GDR_ERR_ALIGN",
                5: "GDR_ERR_WORKSPACE", 6: "GDR_ERR_CUDA", 7: "GDR_ERR_DEVICE_TIMEOUT",
                8: "GDR_ERR_UNSUPPORTED", 9: "GDR_ERR_ARG"}
DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
VARIANTS = {"auto": 0, "simt": 1, "tensor": 2, "fused": 3, "fused_tc": 4}
EXPORTS = ["gdr_prepare_wy", "gdr_scan_h", "gdr_chunk_output", "gdr_forward", "gdr_forward_workspace_bytes",
           "gdr_forward_host", "gdr_forward_host_scratch_bytes",
           "gdr_forward_static_scratch", "gdr_scan_output", "gdr_prepare_wyp", "gdr_gated_operands",
           "gdr_bwd_dv_local", "gdr_bwd_scan_dh", "gdr_bwd_dqkwg", "gdr_bwd_wy", "gdr_backward",
           "gdr_backward_workspace_bytes", "gdr_bwd_prepare", "gdr_bwd_scan_dh_p", "gdr_bwd_wy_dqkg",
           "gdr_bwd_group_sum", "gdr_bwd_dv_local_tc", "gdr_bwd_scan_dh_tc", "gdr_scan_transfer",
           "gdr_scan_combine", "gdr_scan_combine_reverse", "gdr_forward_segments",
           "gdr_varlen_forward", "gdr_varlen_forward_workspace_bytes", "gdr_varlen_backward",
           "gdr_varlen_backward_workspace_bytes",
           "gdr_status_string", "gdr_get_device_status", "gdr_selftest_bounded_wait", "gdr_last_variant",
           "gdr_version"]


class GdrError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({_status_text(status)})")


class gdr_problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("H", ctypes.c_int64), ("K", ctypes.c_int64),
                ("V", ctypes.c_int64), ("chunk", ctypes.c_int64), ("io_dtype", ctypes.c_int32),
                ("gate", ctypes.c_int32), ("scale", ctypes.c_float), ("variant", ctypes.c_int32),
                ("HV", ctypes.c_int64), ("segments", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def load(path: str | None = None):
    """Load libgdr.so (built by `build.py`).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libgdr is not built ({p} missing); run __graft_entry__.build() "
                               "or python -m chunked_gated_delta_prepare_gb300.build")
        lib = ctypes.CDLL(p)
        vp, P = ctypes.c_void_p, ctypes.POINTER(gdr_problem)
        sig = {
            "gdr_prepare_wy": [P, vp, vp, vp, vp, vp, vp, vp, vp],
            "gdr_scan_h": [P, vp, vp, vp, vp, vp, vp, vp, vp, vp],
            "gdr_chunk_output": [P, vp, vp, vp, vp, vp, vp, vp],
            "gdr_forward": [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp],
            "gdr_forward_static_scratch": [P, vp, vp, vp, vp, vp, vp, vp, vp, vp],
            "gdr_scan_output": [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp],
            "gdr_prepare_wyp": [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp],
            "gdr_gated_operands": [P, vp, vp, vp, vp, vp, vp, vp],
            "gdr_forward_workspace_bytes": [P],
            "gdr_forward_host": [P, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int32, vp, ctypes.c_size_t, vp],
            "gdr_forward_host_scratch_bytes": [P, ctypes.c_int32],
            "gdr_bwd_dv_local": [P, vp, vp, vp, vp, vp, vp],
            "gdr_bwd_scan_dh": [P] + [vp] * 11,
            "gdr_bwd_dqkwg": [P] + [vp] * 14,
            "gdr_bwd_wy": [P] + [vp] * 14,
            "gdr_backward": [P] + [vp] * 15 + [ctypes.c_size_t, vp],
            "gdr_backward_workspace_bytes": [P],
            "gdr_bwd_prepare": [P] + [vp] * 11,
            "gdr_bwd_scan_dh_p": [P] + [vp] * 11,
            "gdr_bwd_wy_dqkg": [P] + [vp] * 20,
            "gdr_bwd_group_sum": [P] + [vp] * 5,
            "gdr_bwd_dv_local_tc": [P] + [vp] * 6,
            "gdr_bwd_scan_dh_tc": [P] + [vp] * 11,
            "gdr_scan_transfer": [P, vp, vp, vp, vp, ctypes.c_int32, vp, vp, vp],
            "gdr_scan_combine": [P, ctypes.c_int32, vp, vp, vp, vp, vp, vp],
            "gdr_scan_combine_reverse": [P, ctypes.c_int32, vp, vp, vp, vp, vp, vp],
            "gdr_forward_segments": [P],
            "gdr_varlen_forward": [P, vp, vp, ctypes.c_int64] + [vp] * 8 + [vp, ctypes.c_size_t, vp],
            "gdr_varlen_forward_workspace_bytes": [P],
            "gdr_varlen_backward": [P, vp, vp, ctypes.c_int64] + [vp] * 14 + [vp, ctypes.c_size_t, vp],
            "gdr_varlen_backward_workspace_bytes": [P],
            "gdr_status_string": [ctypes.c_int],
            "gdr_get_device_status": [vp],
            "gdr_selftest_bounded_wait": [ctypes.c_int32, ctypes.c_int32, vp],
            "gdr_last_variant": [],
            "gdr_version": [],
        }
        for name, args in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        lib.gdr_forward_workspace_bytes.restype = ctypes.c_size_t
        lib.gdr_forward_host_scratch_bytes.restype = ctypes.c_size_t
        lib.gdr_backward_workspace_bytes.restype = ctypes.c_size_t
        lib.gdr_varlen_forward_workspace_bytes.restype = ctypes.c_size_t
        lib.gdr_varlen_backward_workspace_bytes.restype = ctypes.c_size_t
        lib.gdr_status_string.restype = ctypes.c_char_p
        lib.gdr_last_variant.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def _status_text(status: int) -> str:
    try:
        return load().gdr_status_string(status).decode()
    except Exception:  # the library may be the thing that is missing
        return "?"


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != GDR_OK:
        raise GdrError(status, where)


def make_problem(B, T, H, K, V, chunk, io_dtype=torch.bfloat16, per_k_gate=False, scale=None,
                 variant="auto", HV=0, segments=0) -> gdr_problem:
    """H: q/k heads; HV: value heads (a multiple of H; 0 means H); segments: gdr_forward's
    segment-parallel scan (0 = the library's choice, 1 = off, S = S segments)."""
    dt = DTYPES[io_dtype] if isinstance(io_dtype, torch.dtype) else int(io_dtype)
    return gdr_problem(B=B, T=T, H=H, K=K, V=V, chunk=chunk, io_dtype=dt, gate=1 if per_k_gate else 0,
                       scale=-1.0 if scale is None else float(scale),
                       variant=VARIANTS[variant] if isinstance(variant, str) else int(variant), HV=HV,
                       segments=int(segments))


def problem_for(q, v, g, chunk, scale=None, variant="auto", segments=0) -> gdr_problem:
    """The problem of tensors q [B,T,H,K], v [B,T,HV,V] and g; HV > H means grouped value heads."""
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[-1]
    return make_problem(B, T, H, K, V, chunk, q.dtype, g.dim() == 4, scale, variant, HV=HV if HV != H else 0,
                        segments=segments)


# ---------------------------------------------------------------- raw entry points

def gdr_prepare_wy(p, k, v, g, beta, w, u, g_cum, stream=None):
    _check(load().gdr_prepare_wy(ctypes.byref(p), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(w), _ptr(u),
                                 _ptr(g_cum), _stream(stream)), "gdr_prepare_wy")


def gdr_scan_transfer(p, k, w, u, g_cum, segments, M, Z, stream=None):
    _check(load().gdr_scan_transfer(ctypes.byref(p), _ptr(k), _ptr(w), _ptr(u), _ptr(g_cum), int(segments), _ptr(M),
                                    _ptr(Z), _stream(stream)), "gdr_scan_transfer")


def gdr_scan_combine(p, segments, M, Z, h0, h_start, h_final, stream=None):
    _check(load().gdr_scan_combine(ctypes.byref(p), int(segments), _ptr(M), _ptr(Z), _ptr(h0), _ptr(h_start),
                                   _ptr(h_final), _stream(stream)), "gdr_scan_combine")


def gdr_scan_combine_reverse(p, segments, M, Zb, dh_final, ends, dh0, stream=None):
    _check(load().gdr_scan_combine_reverse(ctypes.byref(p), int(segments), _ptr(M), _ptr(Zb), _ptr(dh_final),
                                           _ptr(ends), _ptr(dh0), _stream(stream)), "gdr_scan_combine_reverse")


def gdr_forward_segments(p) -> int:
    return int(load().gdr_forward_segments(ctypes.byref(p)))


def gdr_scan_h(p, k, w, u, g_cum, h0, h_ckpt, v_new, h_final, stream=None):
    _check(load().gdr_scan_h(ctypes.byref(p), _ptr(k), _ptr(w), _ptr(u), _ptr(g_cum), _ptr(h0), _ptr(h_ckpt),
                             _ptr(v_new), _ptr(h_final), _stream(stream)), "gdr_scan_h")


def gdr_chunk_output(p, q, k, v_new, h_ckpt, g_cum, o, stream=None):
    _check(load().gdr_chunk_output(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v_new), _ptr(h_ckpt), _ptr(g_cum),
                                   _ptr(o), _stream(stream)), "gdr_chunk_output")


def gdr_scan_output(p, q, k, w, u, g_cum, P, h0, o, h_final, stream=None):
    _check(load().gdr_scan_output(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(w), _ptr(u), _ptr(g_cum), _ptr(P),
                                  _ptr(h0), _ptr(o), _ptr(h_final), _stream(stream)), "gdr_scan_output")


def gdr_prepare_wyp(p, q, k, v, g, beta, w, u, g_cum, P, stream=None):
    _check(load().gdr_prepare_wyp(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(w), _ptr(u),
                                  _ptr(g_cum), _ptr(P), _stream(stream)), "gdr_prepare_wyp")


def gdr_forward_workspace_bytes(p) -> int:
    return int(load().gdr_forward_workspace_bytes(ctypes.byref(p)))


def gdr_forward(p, q, k, v, g, beta, h0, o, h_final, workspace, workspace_bytes, stream=None):
    _check(load().gdr_forward(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o),
                              _ptr(h_final), _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "gdr_forward")


def gdr_gated_operands(p, q, k, g_cum, P, kg, qg, stream=None):
    _check(load().gdr_gated_operands(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(g_cum), _ptr(P), _ptr(kg), _ptr(qg),
                                     _stream(stream)), "gdr_gated_operands")


def gdr_forward_host_scratch_bytes(p, pieces=0) -> int:
    return int(load().gdr_forward_host_scratch_bytes(ctypes.byref(p), int(pieces)))


def gdr_forward_host(p, q, k, v, g, beta, h0, o, h_final, pieces, scratch, scratch_bytes, stream=None):
    """gdr_forward over host tensors (q .. beta, h0 in, o and h_final out, all host memory), pipelined
    against the host link inside the library (see include/gdr.h)."""
    _check(load().gdr_forward_host(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                   _ptr(o), _ptr(h_final), int(pieces), _ptr(scratch), int(scratch_bytes),
                                   _stream(stream)), "gdr_forward_host")


def gdr_forward_static_scratch(p, q, k, v, g, beta, h0, o, h_final, stream=None):
    """gdr_forward with the scratch taken from the library's fixed device array
    (for callers that cannot allocate device memory; see include/gdr.h)."""
    _check(load().gdr_forward_static_scratch(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                             _ptr(h0), _ptr(o), _ptr(h_final), _stream(stream)),
           "gdr_forward_static_scratch")


STATIC_SCRATCH_BYTES = 64 << 20


def gdr_status_string(status: int) -> str:
    return load().gdr_status_string(int(status)).decode()


def gdr_get_device_status(stream=None) -> int:
    return int(load().gdr_get_device_status(_stream(stream)))


def gdr_selftest_bounded_wait(polls: int, arrive: bool, stream=None):
    """Run the bounded-wait check: a kernel waits on an mbarrier with a limit of `polls` polls;
    with arrive=False nothing arrives and the wait gives up (see include/gdr.h)."""
    _check(load().gdr_selftest_bounded_wait(int(polls), 1 if arrive else 0, _stream(stream)),
           "gdr_selftest_bounded_wait")


def gdr_last_variant() -> str:
    return load().gdr_last_variant().decode()


def gdr_version() -> int:
    return int(load().gdr_version())


# ---------------------------------------------------------------- convenience

def _forward_host(q, k, v, g, beta, h0, chunk, scale, variant, want_h_final, stream, segments, out, h_final_out,
                  pieces, workspace):
    """forward() for host tensors through gdr_forward_host: the library runs the sequence in token pieces
    of whole chunks and overlaps each piece's copies with the computation of its neighbours, carrying the
    fp32 state between pieces, so the results are those of one call over the whole sequence."""
    dev = torch.device("cuda", torch.cuda.current_device())
    B, T, _, K = q.shape
    H, V = v.shape[2], v.shape[-1]
    srcs = [t.contiguous() for t in (q, k, v, g, beta)]
    h0 = h0.contiguous() if h0 is not None else None
    p = problem_for(q, v, g, chunk, scale, variant, segments)
    o = out if out is not None else torch.empty(B, T, H, V, dtype=q.dtype, pin_memory=True)
    hf = None
    if want_h_final:
        hf = h_final_out if h_final_out is not None else torch.empty(B, H, K, V, dtype=torch.float32, pin_memory=True)
    nbytes = gdr_forward_host_scratch_bytes(p, pieces)
    ws = workspace
    if ws is None or not ws.is_cuda or ws.numel() * ws.element_size() < nbytes:
        ws = torch.empty(nbytes, device=dev, dtype=torch.uint8)
    gdr_forward_host(p, *srcs, h0, o, hf, pieces, ws, ws.numel() * ws.element_size(), stream)
    (torch.cuda.current_stream() if stream is None else stream).synchronize()
    return o, hf


def forward(q, k, v, g, beta, h0=None, *, chunk=64, scale=None, variant="auto", want_h_final=True,
            workspace=None, stream=None, segments=0, out=None, h_final_out=None, pieces=8):
    """o, h_final = forward(q, k, v, g, beta, h0).

    Device tensors are used in place.  CPU tensors (pinned for asynchronous
    copies) go to the current CUDA device and the results come back: into `out`
    / `h_final_out` when given (host tensors of o's and h_final's shape and
    dtype), else into new pinned host tensors.  Host inputs go through
    gdr_forward_host in `pieces` token ranges of whole chunks, so the copies
    overlap the kernels (pieces=1: one copy in, one call, one copy out).  The
    results are complete on return.
    """
    on_host = q.device.type == "cpu"
    if on_host and pieces > 1 and -(-q.shape[1] // chunk) >= 2:
        return _forward_host(q, k, v, g, beta, h0, chunk, scale, variant, want_h_final, stream, segments, out,
                             h_final_out, pieces, workspace)
    if on_host:
        dev = torch.device("cuda", torch.cuda.current_device())
        q, k, v, g, beta = (t.to(dev, non_blocking=True) for t in (q, k, v, g, beta))
        h0 = h0.to(dev, non_blocking=True) if h0 is not None else None
    p = problem_for(q, v, g, chunk, scale, variant, segments)
    B, T, _, K = q.shape
    H, V = v.shape[2], v.shape[-1]            # value heads
    o = torch.empty(B, T, H, V, device=q.device, dtype=q.dtype)
    hf = torch.empty(B, H, K, V, device=q.device, dtype=torch.float32) if want_h_final else None
    nbytes = gdr_forward_workspace_bytes(p)
    if workspace is None and nbytes:
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    # the size handed to the library is what the buffer really holds; the library
    # refuses (GDR_ERR_WORKSPACE) a buffer smaller than this problem needs
    have = 0 if workspace is None else workspace.numel() * workspace.element_size()
    gdr_forward(p, q, k, v, g, beta, h0, o, hf, workspace, have, stream)
    if on_host:
        if out is not None:
            out.copy_(o, non_blocking=True)
            o = out
        else:
            o = o.to("cpu")
        if hf is not None:
            if h_final_out is not None:
                h_final_out.copy_(hf, non_blocking=True)
                hf = h_final_out
            else:
                hf = hf.to("cpu")
        torch.cuda.current_stream().synchronize()   # the results are on the host when this returns
    return o, hf


def gdr_bwd_dv_local(p, q, k, g_cum, d_o, dv_loc, stream=None):
    _check(load().gdr_bwd_dv_local(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(g_cum), _ptr(d_o), _ptr(dv_loc),
                                   _stream(stream)), "gdr_bwd_dv_local")


def gdr_bwd_scan_dh(p, q, k, w, g_cum, d_o, dv_loc, dh_final, dh_ckpt, dv_new, dh0, stream=None):
    _check(load().gdr_bwd_scan_dh(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(w), _ptr(g_cum), _ptr(d_o),
                                  _ptr(dv_loc), _ptr(dh_final), _ptr(dh_ckpt), _ptr(dv_new), _ptr(dh0),
                                  _stream(stream)), "gdr_bwd_scan_dh")


def gdr_bwd_dqkwg(p, q, k, v_new, g_cum, h_ckpt, dh_ckpt, d_o, dv_new, dq, dk_part, dw, dG_part, only=None,
                  stream=None):
    _check(load().gdr_bwd_dqkwg(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v_new), _ptr(g_cum), _ptr(h_ckpt),
                                _ptr(dh_ckpt), _ptr(d_o), _ptr(dv_new), _ptr(dq), _ptr(dk_part), _ptr(dw),
                                _ptr(dG_part), _ptr(only), _stream(stream)), "gdr_bwd_dqkwg")


def gdr_bwd_wy(p, k, v, beta, g_cum, dw, dv_new, dk_part, dG_part, dk, dv, dbeta, dg, only=None, stream=None):
    _check(load().gdr_bwd_wy(ctypes.byref(p), _ptr(k), _ptr(v), _ptr(beta), _ptr(g_cum), _ptr(dw), _ptr(dv_new),
                             _ptr(dk_part), _ptr(dG_part), _ptr(dk), _ptr(dv), _ptr(dbeta), _ptr(dg), _ptr(only),
                             _stream(stream)), "gdr_bwd_wy")


def gdr_bwd_prepare(p, q, k, v, g, beta, w, u, g_cum, P, tinv, stream=None):
    _check(load().gdr_bwd_prepare(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(w), _ptr(u),
                                  _ptr(g_cum), _ptr(P), _ptr(tinv), _stream(stream)), "gdr_bwd_prepare")


def gdr_bwd_scan_dh_p(p, q, k, w, g_cum, P, d_o, dh_final, dh_ckpt, dv_new, dh0, stream=None):
    _check(load().gdr_bwd_scan_dh_p(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(w), _ptr(g_cum), _ptr(P), _ptr(d_o),
                                    _ptr(dh_final), _ptr(dh_ckpt), _ptr(dv_new), _ptr(dh0), _stream(stream)),
           "gdr_bwd_scan_dh_p")


def gdr_bwd_wy_dqkg(p, q, k, v, beta, g_cum, w, u, tinv, v_new, h_ckpt, d_o, dv_new, dh_ckpt, dq, dk, dv, dbeta, dg,
                    exact_flags=None, stream=None):
    _check(load().gdr_bwd_wy_dqkg(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g_cum), _ptr(w),
                                  _ptr(u), _ptr(tinv), _ptr(v_new), _ptr(h_ckpt), _ptr(d_o), _ptr(dv_new),
                                  _ptr(dh_ckpt), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbeta), _ptr(dg),
                                  _ptr(exact_flags), _stream(stream)), "gdr_bwd_wy_dqkg")


def gdr_bwd_dv_local_tc(p, q, k, g_cum, d_o, dv_loc, stream=None):
    _check(load().gdr_bwd_dv_local_tc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(g_cum), _ptr(d_o), _ptr(dv_loc),
                                      _stream(stream)), "gdr_bwd_dv_local_tc")


def gdr_bwd_scan_dh_tc(p, q, k, w, g_cum, dv_loc, d_o, dh_final, dh_ckpt, dv_new, dh0, stream=None):
    _check(load().gdr_bwd_scan_dh_tc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(w), _ptr(g_cum), _ptr(dv_loc), _ptr(d_o),
                                     _ptr(dh_final), _ptr(dh_ckpt), _ptr(dv_new), _ptr(dh0), _stream(stream)),
           "gdr_bwd_scan_dh_tc")


def gdr_bwd_group_sum(p, dq_v, dk_v, dq, dk, stream=None):
    _check(load().gdr_bwd_group_sum(ctypes.byref(p), _ptr(dq_v), _ptr(dk_v), _ptr(dq), _ptr(dk), _stream(stream)),
           "gdr_bwd_group_sum")


def gdr_backward_workspace_bytes(p) -> int:
    return int(load().gdr_backward_workspace_bytes(ctypes.byref(p)))


def gdr_backward(p, q, k, v, g, beta, h0, d_o, dh_final, dq, dk, dv, dg, dbeta, dh0, workspace, workspace_bytes,
                 stream=None):
    _check(load().gdr_backward(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                               _ptr(d_o), _ptr(dh_final), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta),
                               _ptr(dh0), _ptr(workspace), int(workspace_bytes), _stream(stream)), "gdr_backward")


def backward(q, k, v, g, beta, h0, d_o, dh_final=None, *, chunk=64, scale=None, variant="auto", workspace=None,
             stream=None, segments=0):
    """dq, dk, dv, dg, dbeta, dh0 = backward(q, k, v, g, beta, h0, do, dh_final): the gradient of
    forward's (o, h_final) against do and dh_final, on device tensors."""
    p = problem_for(q, v, g, chunk, scale, variant, segments)
    B, T, _, K = q.shape
    H, V = v.shape[2], v.shape[-1]            # value heads
    dq, dk = torch.empty_like(q), torch.empty_like(k)
    dv = torch.empty_like(v)
    dg = torch.empty_like(g)
    dbeta = torch.empty_like(beta)
    dh0 = torch.empty(B, H, K, V, device=q.device, dtype=torch.float32)
    nbytes = gdr_backward_workspace_bytes(p)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), device=q.device, dtype=torch.uint8)
    have = workspace.numel() * workspace.element_size()
    gdr_backward(p, q, k, v, g, beta, h0, d_o, dh_final, dq, dk, dv, dg, dbeta, dh0, workspace, have, stream)
    return dq, dk, dv, dg, dbeta, dh0


# ---------------------------------------------------------------- packed variable-length sequences

def gdr_varlen_forward_workspace_bytes(p) -> int:
    return int(load().gdr_varlen_forward_workspace_bytes(ctypes.byref(p)))


def gdr_varlen_backward_workspace_bytes(p) -> int:
    return int(load().gdr_varlen_backward_workspace_bytes(ctypes.byref(p)))


def _host_cu(cu):
    """cu_seqlens as a contiguous host int32 tensor (and its pointer for the C ABI)."""
    if isinstance(cu, torch.Tensor):
        h = cu.detach().to("cpu", torch.int32).contiguous()
    else:
        h = torch.tensor(list(cu), dtype=torch.int32)
    return h


def gdr_varlen_forward(p, cu_seqlens, cu_seqlens_device, total, q, k, v, g, beta, h0, o, h_final, workspace,
                       workspace_bytes, stream=None):
    """cu_seqlens: a host int32 tensor [n + 1]; cu_seqlens_device: a device int32 tensor or None."""
    _check(load().gdr_varlen_forward(ctypes.byref(p), _ptr(cu_seqlens), _ptr(cu_seqlens_device), int(total), _ptr(q),
                                     _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(h_final),
                                     _ptr(workspace), int(workspace_bytes), _stream(stream)), "gdr_varlen_forward")


def gdr_varlen_backward(p, cu_seqlens, cu_seqlens_device, total, q, k, v, g, beta, h0, d_o, dh_final, dq, dk, dv, dg,
                        dbeta, dh0, workspace, workspace_bytes, stream=None):
    _check(load().gdr_varlen_backward(ctypes.byref(p), _ptr(cu_seqlens), _ptr(cu_seqlens_device), int(total),
                                      _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(d_o),
                                      _ptr(dh_final), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dh0),
                                      _ptr(workspace), int(workspace_bytes), _stream(stream)), "gdr_varlen_backward")


def varlen_problem(q, v, g, cu_host, max_len, chunk, scale, variant, segments):
    """The padded problem of packed q [total,H,K] (or [1,total,H,K]), v, g: B = n sequences, T = max_len."""
    n = cu_host.numel() - 1
    if n < 1:
        raise ValueError("cu_seqlens needs at least two entries")
    lens = (cu_host[1:] - cu_host[:-1]).tolist()
    T = max(max(lens), 1) if max_len is None else int(max_len)
    H, K = q.shape[-2], q.shape[-1]
    HV, V = v.shape[-2], v.shape[-1]
    per_k = g.dim() == q.dim()
    return make_problem(n, T, H, K, V, chunk, q.dtype, per_k, scale, variant, HV=HV if HV != H else 0,
                        segments=segments)


def forward_varlen(q, k, v, g, beta, cu_seqlens, h0=None, *, chunk=64, scale=None, variant="auto", max_len=None,
                   want_h_final=True, workspace=None, stream=None, segments=0):
    """o, h_final = forward_varlen(q, k, v, g, beta, cu_seqlens, h0) on packed device tensors.

    q, k [total,H,K] (or with a leading 1), v [total,HV,V], g [total,HV(,K)], beta [total,HV];
    cu_seqlens: the n + 1 cumulative lengths (list, host or device int32 tensor); h0 [n,HV,K,V] or None.
    Returns o packed like v and h_final [n,HV,K,V] fp32 (None if not wanted)."""
    cu_host = _host_cu(cu_seqlens)
    cu_dev = cu_seqlens if (isinstance(cu_seqlens, torch.Tensor) and cu_seqlens.is_cuda
                            and cu_seqlens.dtype == torch.int32 and cu_seqlens.is_contiguous()) else None
    p = varlen_problem(q, v, g, cu_host, max_len, chunk, scale, variant, segments)
    total = int(cu_host[-1])
    n, K, HV, V = int(p.B), q.shape[-1], v.shape[-2], v.shape[-1]
    o = torch.empty(v.shape, device=v.device, dtype=v.dtype)
    hf = torch.empty(n, HV, K, V, device=v.device, dtype=torch.float32) if want_h_final else None
    if workspace is None:
        workspace = torch.empty(max(gdr_varlen_forward_workspace_bytes(p), 1), device=v.device, dtype=torch.uint8)
    have = workspace.numel() * workspace.element_size()
    gdr_varlen_forward(p, cu_host, cu_dev, total, q, k, v, g, beta, h0, o, hf, workspace, have, stream)
    return o, hf


def backward_varlen(q, k, v, g, beta, cu_seqlens, h0, d_o, dh_final=None, *, chunk=64, scale=None, variant="auto",
                    max_len=None, workspace=None, stream=None, segments=0):
    """dq, dk, dv, dg, dbeta, dh0 = backward_varlen(...): the gradient of forward_varlen's (o, h_final)
    against do (packed like o) and dh_final [n,HV,K,V]; packed outputs like their inputs."""
    cu_host = _host_cu(cu_seqlens)
    cu_dev = cu_seqlens if (isinstance(cu_seqlens, torch.Tensor) and cu_seqlens.is_cuda
                            and cu_seqlens.dtype == torch.int32 and cu_seqlens.is_contiguous()) else None
    p = varlen_problem(q, v, g, cu_host, max_len, chunk, scale, variant, segments)
    total = int(cu_host[-1])
    n, K, HV, V = int(p.B), q.shape[-1], v.shape[-2], v.shape[-1]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg, dbeta = torch.empty_like(g), torch.empty_like(beta)
    dh0 = torch.empty(n, HV, K, V, device=v.device, dtype=torch.float32)
    if workspace is None:
        workspace = torch.empty(max(gdr_varlen_backward_workspace_bytes(p), 1), device=v.device, dtype=torch.uint8)
    have = workspace.numel() * workspace.element_size()
    gdr_varlen_backward(p, cu_host, cu_dev, total, q, k, v, g, beta, h0, d_o, dh_final, dq, dk, dv, dg, dbeta, dh0,
                        workspace, have, stream)
    return dq, dk, dv, dg, dbeta, dh0


def default_scale(K: int) -> float:
    return 1.0 / math.sqrt(K)
