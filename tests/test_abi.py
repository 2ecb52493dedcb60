"""Host-side checks of the C ABI: the library builds and loads without a GPU,
exports every function include/gdr.h declares, and rejects bad arguments with
the documented status codes before it launches anything."""
import ctypes
import os
import re
import threading

import pytest

from chunked_gated_delta_prepare_gb300 import build as gdr_build
from chunked_gated_delta_prepare_gb300 import gdr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdr.h")


@pytest.fixture(scope="module")
def lib():
    gdr_build.build()
    return gdr.load()


def declared_functions():
    with open(HEADER) as f:
        src = f.read()
    return re.findall(r"^GDR_API\s+[\w\s\*]+?\b(gdr_\w+)\s*\(", src, flags=re.M)


def test_header_declares_the_stage_entry_points():
    names = declared_functions()
    for n in ("gdr_prepare_wy", "gdr_scan_h", "gdr_chunk_output", "gdr_forward", "gdr_forward_workspace_bytes",
              "gdr_status_string", "gdr_get_device_status", "gdr_last_variant", "gdr_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(gdr.EXPORTS) <= set(declared_functions())


def declared_arity():
    """name -> number of parameters, from the prototypes in include/gdr.h."""
    with open(HEADER) as f:
        src = f.read()
    out = {}
    for m in re.finditer(r"^GDR_API\s+[\w\s\*]+?\b(gdr_\w+)\s*\(([^)]*)\)", src, flags=re.M):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else len(params.split(","))
    return out


def test_binding_arity_matches_the_header(lib):
    arity = declared_arity()
    assert len(arity) == len(declared_functions())
    for name, n in arity.items():
        assert len(getattr(lib, name).argtypes) == n, name


def test_status_strings(lib):
    for code in range(10):
        s = gdr.gdr_status_string(code)
        assert s and s != "unknown status"
    assert gdr.gdr_status_string(123) == "unknown status"


def test_last_variant_empty_on_new_thread(lib):
    out = []
    t = threading.Thread(target=lambda: out.append(gdr.gdr_last_variant()))
    t.start()
    t.join()
    assert out == [""]


def _fwd(lib, p, ptrs=None, ws=None, ws_bytes=0):
    a = dict(q=16, k=16, v=16, g=16, beta=16, h0=None, o=16, hf=None)
    a.update(ptrs or {})
    return lib.gdr_forward(ctypes.byref(p) if p is not None else None, a["q"], a["k"], a["v"], a["g"], a["beta"],
                           a["h0"], a["o"], a["hf"], ws, ws_bytes, None)


def good():
    return gdr.make_problem(1, 256, 2, 64, 64, 64)


@pytest.mark.parametrize("field,value,code", [
    ("T", 0, 2), ("T", -5, 2), ("B", 0, 2), ("H", -1, 2), ("K", 96, 2), ("V", 32, 2), ("chunk", 16, 2),
    ("chunk", 0, 2), ("H", 70000, 2), ("io_dtype", 7, 3), ("gate", 2, 3), ("variant", 9, 9),
    ("scale", float("nan"), 9), ("scale", float("inf"), 9),
])
def test_bad_problem_is_rejected(lib, field, value, code):
    p = good()
    setattr(p, field, value)
    assert _fwd(lib, p) == code
    assert lib.gdr_forward_workspace_bytes(ctypes.byref(p)) == 0


def test_null_problem(lib):
    assert _fwd(lib, None) == 1
    assert lib.gdr_forward_workspace_bytes(None) == 0


@pytest.mark.parametrize("name", ["q", "k", "v", "g", "beta", "o"])
def test_null_required_pointer(lib, name):
    assert _fwd(lib, good(), {name: None}) == 1


@pytest.mark.parametrize("name", ["q", "k", "v", "g", "beta", "o", "h0", "hf"])
def test_misaligned_pointer(lib, name):
    assert _fwd(lib, good(), {name: 24}) == 4


def test_workspace_checks(lib):
    p = good()
    need = lib.gdr_forward_workspace_bytes(ctypes.byref(p))
    assert need > 0
    assert _fwd(lib, p, ws=None, ws_bytes=need) == 5
    assert _fwd(lib, p, ws=256, ws_bytes=need - 1) == 5
    assert _fwd(lib, p, ws=272, ws_bytes=need) == 4          # workspace must be 256-byte aligned


def test_workspace_size_formula(lib):
    # g_cum fp32, then w, u, v_new, h_ckpt in the io dtype, each rounded up to 256 bytes
    for (B, T, H, K, V, C, bf16, per_k) in [(1, 256, 2, 64, 64, 64, 0, 0), (2, 4096, 8, 64, 64, 32, 1, 0),
                                            (2, 8192, 16, 128, 128, 64, 1, 1)]:
        p = gdr.make_problem(B, T, H, K, V, C, 1 if bf16 else 0, bool(per_k), variant="simt")
        e = 2 if bf16 else 4
        r = lambda x: (x + 255) // 256 * 256
        rows = B * T * H
        want = r(rows * (K if per_k else 1) * 4) + r(rows * K * e) + 2 * r(rows * V * e) + r(B * (T // C) * H * K * V * e)
        assert lib.gdr_forward_workspace_bytes(ctypes.byref(p)) == want


def test_partial_last_chunk_is_accepted_and_checkpointed():
    # T = 100 with 64-token chunks: two chunks, the second one partial, each with a checkpoint
    r = lambda x: (x + 255) // 256 * 256
    p = gdr.make_problem(2, 100, 3, 64, 128, 64, 1, False, variant="tensor")
    rows = 2 * 100 * 3
    want = r(rows * 4) + r(rows * 64 * 2) + 2 * r(rows * 128 * 2) + r(2 * 2 * 3 * 64 * 128 * 2)
    assert lib_bytes(p) == want
    # the fused path's gated scores are per chunk: [B, NT, H, C, C]
    p = gdr.make_problem(2, 100, 3, 64, 128, 64, 1, False, variant="fused")
    assert lib_bytes(p) == r(rows * 4) + r(rows * 64 * 2) + r(rows * 128 * 2) + r(2 * 2 * 3 * 64 * 64 * 2)
    for T in (1, 31, 33, 65):
        assert lib_bytes(gdr.make_problem(1, T, 1, 64, 64, 32, 0, True, variant="simt")) > 0


def lib_bytes(p):
    return gdr.load().gdr_forward_workspace_bytes(ctypes.byref(p))


def test_fused_workspace_size_formula(lib):
    # g_cum, w, u, then (64-token chunks) the gated scores P [B, NT, H, 64, 64] bf16; no v_new or checkpoints
    r = lambda x: (x + 255) // 256 * 256
    for (B, T, H, K, V, C) in [(1, 256, 2, 64, 64, 64), (2, 4096, 8, 64, 64, 32), (1, 32768, 32, 128, 128, 64)]:
        rows = B * T * H
        want = r(rows * 4) + r(rows * K * 2) + r(rows * V * 2) + (r(rows * C * 2) if C == 64 else 0)
        variants = ["fused", "auto" if C == 64 else "fused"]
        if K == V == 128 and C == 64 and B > 1:
            variants.append("fused_tc")      # the tcgen05 form keeps the same intermediates (batched: no pieces)
        for variant in variants:
            p = gdr.make_problem(B, T, H, K, V, C, 1, False, variant=variant, segments=1)
            extra = 0
            if variant == "auto" and B == 1 and K == V == 128 and -(-T // C) >= 128:
                # AUTO runs one long sequence on the overlapped tcgen05 path: 7 pieces here, the state carried
                # between them in fp32
                extra = r((overlap_pieces(-(-T // C)) - 1) * H * K * V * 4)
            assert lib.gdr_forward_workspace_bytes(ctypes.byref(p)) == want + extra


def overlap_pieces(NT, first=16, most=32):
    """The overlapped forward's piece count for NT chunks: sizes grow from 16 chunks by 3/2, never below an
    equal share of what is left among the pieces still allowed (at most 32); none below 128 chunks."""
    if NT < 128:
        return 1
    n = c = 0
    ln = first
    while c < NT:
        ln = max(ln, -(-(NT - c) // (most - n)))
        c = min(NT, c + ln)
        n += 1
        ln += ln // 2
    return n


def test_overlap_piece_rule():
    assert [overlap_pieces(n) for n in (64, 127, 128, 131, 193, 512, 2560, 100000)] == [1, 1, 4, 5, 5, 7, 7, 7]


def test_overlapped_fused_tc_workspace(lib):
    # one sequence on the tcgen05 fused path runs in pieces; the workspace adds the fp32 state carried
    # between pieces, [pieces - 1][H, K, V]
    r = lambda x: (x + 255) // 256 * 256
    for (T, H) in [(64 * 64, 2), (64 * 128, 2), (64 * 131 - 10, 3), (32768, 32), (64 * 2560, 1)]:
        rows = T * H
        NT = -(-T // 64)
        pieces = overlap_pieces(NT)
        base = r(rows * 4) + r(rows * 128 * 2) + r(rows * 128 * 2) + r(NT * H * 64 * 64 * 2)
        want = base + (r((pieces - 1) * H * 128 * 128 * 4) if pieces > 1 else 0)
        p = gdr.make_problem(1, T, H, 128, 128, 64, 1, False, variant="fused_tc", segments=1)
        assert lib.gdr_forward_workspace_bytes(ctypes.byref(p)) == want, (T, H)
        # two sequences run batched, not in pieces: no carried state
        rows2 = 2 * rows
        base2 = r(rows2 * 4) + r(rows2 * 128 * 2) + r(rows2 * 128 * 2) + r(2 * NT * H * 64 * 64 * 2)
        p2 = gdr.make_problem(2, T, H, 128, 128, 64, 1, False, variant="fused_tc", segments=1)
        assert lib.gdr_forward_workspace_bytes(ctypes.byref(p2)) == base2


def test_fused_tc_variant_takes_its_sizes_only(lib):
    # K = V = 128, C = 64: bf16 with either gate, fp16 with a scalar gate; anything else is
    # GDR_ERR_UNSUPPORTED before a launch
    for (K, V, C, dt, per_k, code) in [(128, 128, 64, 1, False, None), (64, 64, 64, 1, False, 8),
                                       (128, 64, 64, 1, False, 8), (128, 128, 32, 1, False, 8),
                                       (128, 128, 64, 1, True, None), (128, 128, 32, 1, True, 8),
                                       (128, 128, 64, 0, False, 8), (128, 128, 64, 2, False, None),
                                       (128, 128, 64, 2, True, 8), (64, 64, 64, 2, False, 8),
                                       (128, 128, 32, 2, False, 8)]:
        p = gdr.make_problem(1, 256, 2, K, V, C, dt, per_k, variant="fused_tc")
        if code is None:
            assert lib.gdr_forward_workspace_bytes(ctypes.byref(p)) > 0
        else:
            assert lib.gdr_forward_workspace_bytes(ctypes.byref(p)) == 0
            assert _fwd(lib, p) == code
    p = gdr.make_problem(1, 256, 2, 128, 128, 64, 1, False)
    p.variant = 5
    assert _fwd(lib, p) == 9


def test_fp16_fused_tc_rules(lib):
    # fp16 on the tensor-core paths: no segmented scan; AUTO takes the fused forms at K = V = 128, C = 64
    # with a scalar gate, grouped value heads included (the same workspace as the variant asked by name),
    # and the staged kernels for a per-key-dim gate
    p = gdr.make_problem(1, 256, 2, 128, 128, 64, 2, False, variant="fused_tc", HV=4)
    assert lib.gdr_forward_workspace_bytes(ctypes.byref(p)) == lib.gdr_forward_workspace_bytes(
        ctypes.byref(gdr.make_problem(1, 256, 2, 128, 128, 64, 2, False, HV=4))) > 0
    p = gdr.make_problem(1, 4096, 2, 128, 128, 64, 2, False, variant="fused_tc", segments=4)
    assert lib.gdr_forward_workspace_bytes(ctypes.byref(p)) == 0 and _fwd(lib, p) == 8
    assert lib.gdr_forward_segments(ctypes.byref(gdr.make_problem(1, 4096, 1, 128, 128, 64, 2, False))) == 1
    for B, T in [(2, 320), (1, 64 * 200)]:
        named = gdr.make_problem(B, T, 2, 128, 128, 64, 2, False, variant="fused_tc")
        auto = gdr.make_problem(B, T, 2, 128, 128, 64, 2, False)
        assert lib.gdr_forward_workspace_bytes(ctypes.byref(auto)) == lib.gdr_forward_workspace_bytes(
            ctypes.byref(named)) > 0
    auto = gdr.make_problem(2, 320, 2, 128, 128, 64, 2, True)
    staged = gdr.make_problem(2, 320, 2, 128, 128, 64, 2, True, variant="tensor")
    assert lib.gdr_forward_workspace_bytes(ctypes.byref(auto)) == lib.gdr_forward_workspace_bytes(
        ctypes.byref(staged)) > 0
    # the staged and warp-level variants take fp16 at every shape; the warp-level one a scalar gate only
    for (K, V, C, per_k, variant, ok) in [(64, 64, 32, False, "tensor", True), (64, 128, 64, True, "tensor", True),
                                          (128, 64, 64, False, "fused", True), (64, 64, 32, False, "fused", True),
                                          (64, 64, 64, True, "fused", False)]:
        p = gdr.make_problem(1, 256, 2, K, V, C, 2, per_k, variant=variant)
        if ok:
            assert lib.gdr_forward_workspace_bytes(ctypes.byref(p)) > 0
        else:
            assert lib.gdr_forward_workspace_bytes(ctypes.byref(p)) == 0 and _fwd(lib, p) == 8


def test_fp16_plans_like_bf16(lib):
    # fp16 runs the forward kernels bf16 runs, so every variant plans the same scratch for both, batched
    # and packed, wherever no segmented scan applies; the exceptions are the tcgen05 form with a
    # per-key-dim gate (fp16 refused; AUTO runs the staged kernels there instead, as TENSOR does for
    # bf16) and the segments AUTO picks for bf16 only
    fwd = lambda p: lib.gdr_forward_workspace_bytes(ctypes.byref(p))
    packed = lambda p: lib.gdr_varlen_forward_workspace_bytes(ctypes.byref(p))
    for (B, T, H, K, V, C) in [(4, 320, 16, 128, 128, 64), (4, 300, 16, 64, 64, 32), (4, 200, 16, 128, 64, 64),
                               (4, 256, 16, 64, 128, 32), (1, 64 * 140, 40, 128, 128, 64)]:
        for per_k in (False, True):
            for variant in ("auto", "simt", "tensor", "fused", "fused_tc"):
                b = gdr.make_problem(B, T, H, K, V, C, 1, per_k, variant=variant)
                f = gdr.make_problem(B, T, H, K, V, C, 2, per_k, variant=variant)
                if variant == "fused_tc" and per_k:
                    assert fwd(f) == 0 and (fwd(b) > 0) == (K == V == 128 and C == 64)
                    continue
                if fwd(b) == 0:   # a variant that takes neither (the shape, or a per-key-dim gate)
                    assert fwd(f) == 0 and packed(f) == packed(b) == 0
                    continue
                assert lib.gdr_forward_segments(ctypes.byref(b)) == 1   # no segments: the plans compare
                assert packed(f) == packed(b), (B, T, H, K, V, C, per_k, variant)
                if variant == "auto" and per_k and K == V == 128 and C == 64:
                    b = gdr.make_problem(B, T, H, K, V, C, 1, per_k, variant="tensor")
                assert fwd(f) == fwd(b), (B, T, H, K, V, C, per_k, variant)
    # where AUTO segments a bf16 scan, fp16 scans whole
    b = gdr.make_problem(1, 32768, 4, 128, 128, 64, 1, False)
    f = gdr.make_problem(1, 32768, 4, 128, 128, 64, 2, False)
    assert lib.gdr_forward_segments(ctypes.byref(b)) == 8 and lib.gdr_forward_segments(ctypes.byref(f)) == 1


def test_segment_choice_and_workspace(lib):
    # automatic segments: only when the serial scan's B H V/32 CTAs fill at most half of 152 SMs; the
    # largest divisor S of NT with S B H V/32 <= 152 and NT / S >= 16
    r = lambda x: (x + 255) // 256 * 256
    seg = lambda *a, **kw: lib.gdr_forward_segments(ctypes.byref(gdr.make_problem(*a, **kw)))
    assert seg(1, 32768, 32, 128, 128, 64, 1, False) == 1                   # 128 CTAs: serial
    assert seg(1, 32768, 4, 128, 128, 64, 1, False) == 8                    # 16 CTAs: 152 // 16 = 9 -> 8
    assert seg(2, 4096, 8, 64, 64, 32, 1, False) == 4                       # 32 CTAs, NT = 128
    assert seg(1, 2048, 1, 128, 128, 64, 1, True) == 2                      # NT = 32: segments of 16 chunks
    assert seg(1, 1024, 1, 128, 128, 64, 1, False) == 1                     # too short
    assert seg(1, 32768, 4, 128, 128, 64, 1, False, segments=1) == 1
    assert seg(1, 32768, 4, 128, 128, 64, 1, False, segments=32) == 32     # explicit
    assert seg(1, 32768, 4, 128, 128, 64, 0, False) == 1                    # fp32: the CUDA-core path
    assert seg(1, 32768, 4, 128, 128, 64, 1, False, segments=3) == 0        # does not divide NT
    assert seg(1, 32760, 4, 128, 128, 64, 1, False, segments=2) == 0        # a partial chunk
    assert seg(1, 32768, 4, 128, 128, 64, 1, False, segments=-1) == 0
    B, T, H, K, V, C, S = 1, 32768, 4, 128, 128, 64, 8
    rows = B * T * H
    base = r(rows * 4) + r(rows * K * 2) + r(rows * V * 2) + r(rows * C * 2)
    maps = B * S * H * K
    p = gdr.make_problem(B, T, H, K, V, C, 1, False)
    assert lib.gdr_forward_workspace_bytes(ctypes.byref(p)) == base + r(maps * K * 4) + 2 * r(maps * V * 4)


def test_stage_entry_points_validate(lib):
    p = good()
    P = ctypes.byref(p)
    assert lib.gdr_prepare_wy(P, 16, 16, 16, 16, 16, None, 16, None) == 1
    assert lib.gdr_prepare_wy(P, 16, 16, 16, 16, 16, 16, 20, None) == 4
    assert lib.gdr_scan_h(P, 16, 16, 16, 16, None, None, None, None, None) == 1      # v_new required
    assert lib.gdr_scan_h(P, 16, 16, 16, 16, 8, None, 16, None, None) == 4           # h0 misaligned
    assert lib.gdr_chunk_output(P, 16, 16, 16, None, 16, 16, None) == 1              # h_ckpt required
    p.V = 96
    assert lib.gdr_chunk_output(P, 16, 16, 16, 16, 16, 16, None) == 2


def test_python_binding_raises_on_missing_library(tmp_path):
    with pytest.raises(RuntimeError):
        gdr.load(str(tmp_path / "libgdr_missing.so"))


# ---------------------------------------------------------------- packed variable-length sequences

def _cu(vals):
    return None if vals is None else (ctypes.c_int32 * len(vals))(*vals)


def _varlen_fwd(lib, p, cu, total, cu_dev=None, ws=None, ws_bytes=0, ptrs=None):
    a = dict(q=16, k=16, v=16, g=16, beta=16, h0=None, o=16, hf=None)
    a.update(ptrs or {})
    return lib.gdr_varlen_forward(ctypes.byref(p), _cu(cu), cu_dev, total, a["q"], a["k"], a["v"], a["g"], a["beta"],
                                  a["h0"], a["o"], a["hf"], ws, ws_bytes, None)


def _varlen_bwd(lib, p, cu, total, ws=None, ws_bytes=0):
    return lib.gdr_varlen_backward(ctypes.byref(p), _cu(cu), None, total, 16, 16, 16, 16, 16, None, 16, None, 16, 16,
                                   16, 16, 16, None, ws, ws_bytes, None)


def test_varlen_checks_cu_seqlens_on_the_host(lib):
    p = gdr.make_problem(3, 100, 2, 64, 64, 64)           # three sequences, rows of 100 tokens
    # a good cu reaches the workspace check (no workspace given: GDR_ERR_WORKSPACE) without launching
    assert _varlen_fwd(lib, p, [0, 50, 50, 150], 150) == 5
    assert _varlen_bwd(lib, p, [0, 50, 50, 150], 150) == 5
    assert _varlen_fwd(lib, p, [0, 100, 200, 300], 300) == 5
    for cu, total in (([1, 50, 50, 151], 151),            # does not start at 0
                      ([0, 60, 50, 150], 150),            # decreases
                      ([0, 101, 101, 150], 150),          # a sequence longer than the rows
                      ([0, 50, 50, 150], 149)):           # total is not cu[n]
        assert _varlen_fwd(lib, p, cu, total) == 9, cu
        assert _varlen_bwd(lib, p, cu, total) == 9, cu
    assert _varlen_fwd(lib, p, None, 150) == 1
    assert _varlen_fwd(lib, p, [0, 50, 50, 150], 150, cu_dev=18) == 4   # device cu must be 4-byte aligned
    assert _varlen_fwd(lib, p, [0, 50, 50, 150], 150, ptrs=dict(q=None)) == 1
    assert _varlen_fwd(lib, p, [0, 50, 50, 150], 150, ptrs=dict(o=24)) == 4
    # no tokens at all: the packed pointers may be NULL
    empty = dict(q=None, k=None, v=None, g=None, beta=None, o=None)
    assert _varlen_fwd(lib, p, [0, 0, 0, 0], 0, ptrs=empty) == 5
    p.T = 0
    assert _varlen_fwd(lib, p, [0, 0, 0, 0], 0, ptrs=empty) == 2


def test_varlen_workspace_size_formula(lib):
    # device cu; on the tensor cores also the chunk offsets co [n + 1] and the chunk -> sequence map [NTmax],
    # NTmax = n ceil(T / C); then every working tensor (rows: NTmax C chunk-packed, n T padded), each
    # rounded up to 256 bytes; then the inner call's workspace (on the tensor cores the larger of the padded
    # problem's and that of the largest chunk-packed problem, one row of NTmax chunks; neither segmented)
    r = lambda x: (x + 255) // 256 * 256
    for (n, T, H, HV, K, V, C, dt, per_k, variant) in [(3, 100, 2, 2, 64, 64, 64, 1, False, "auto"),
                                                       (5, 333, 1, 4, 128, 64, 32, 1, True, "auto"),
                                                       (4, 4096, 2, 2, 128, 128, 64, 1, False, "tensor"),
                                                       (2, 64, 2, 2, 64, 128, 64, 0, True, "simt")]:
        mk = lambda B, T_, segments=0: gdr.make_problem(B, T_, H, K, V, C, dt, per_k, variant=variant,
                                                        HV=HV if HV != H else 0, segments=segments)
        p = mk(n, T)
        p1 = mk(n, T, segments=1)      # the padded inner call: each sequence scanned whole
        e = 2 if dt else 4
        qk, vv, gg, bb = H * K * e, HV * V * e, HV * (K if per_k else 1) * 4, HV * e
        chunked = variant != "simt"
        ntmax = n * -(-T // C)
        rows = ntmax * C if chunked else n * T
        head = r((n + 1) * 4) + (r((n + 1) * 4) + r(ntmax * 4) if chunked else 0)
        pad = lambda sizes: sum(r(rows * b) for b in sizes)
        big = mk(1, ntmax * C, segments=1)
        fin = lib.gdr_forward_workspace_bytes(ctypes.byref(p1))
        bin_ = lib.gdr_backward_workspace_bytes(ctypes.byref(p1))
        if chunked:
            fin = max(fin, lib.gdr_forward_workspace_bytes(ctypes.byref(big)))
            bin_ = max(bin_, lib.gdr_backward_workspace_bytes(ctypes.byref(big)))
        fwd = head + pad([qk, qk, vv, gg, bb, vv]) + fin
        bwd = head + pad([qk, qk, vv, gg, bb, vv, qk, qk, vv, gg, bb]) + bin_
        assert lib.gdr_varlen_forward_workspace_bytes(ctypes.byref(p)) == fwd
        assert lib.gdr_varlen_backward_workspace_bytes(ctypes.byref(p)) == bwd
    bad = gdr.make_problem(3, 100, 2, 96, 64, 64)
    assert lib.gdr_varlen_forward_workspace_bytes(ctypes.byref(bad)) == 0
    assert lib.gdr_varlen_backward_workspace_bytes(ctypes.byref(bad)) == 0


def test_varlen_ignores_segments(lib):
    # every sequence is scanned whole: the problem's segment count changes nothing, not even when it would
    # be invalid for the padded batch
    base = gdr.make_problem(4, 4096, 2, 128, 128, 64, 1, False, segments=1)
    for seg in (0, 3, 8):
        p = gdr.make_problem(4, 4096, 2, 128, 128, 64, 1, False, segments=seg)
        for fn in (lib.gdr_varlen_forward_workspace_bytes, lib.gdr_varlen_backward_workspace_bytes):
            assert fn(ctypes.byref(p)) == fn(ctypes.byref(base)) > 0
    assert lib.gdr_varlen_forward_workspace_bytes(None) == 0
    assert lib.gdr_varlen_forward(None, None, None, 0, None, None, None, None, None, None, None, None, None, 0,
                                  None) == 1


def test_header_is_plain_c_and_a_c_program_links(lib, tmp_path):
    # the boundary is a C ABI: a C99 program includes gdr.h, links libgdr and calls the host-only entry
    # points (no device is touched: version, status text, workspace sizes, a validation error)
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_gdr.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "gdr.h"
int main(void) {
    gdr_problem p;
    memset(&p, 0, sizeof p);
    p.B = 2; p.T = 256; p.H = 4; p.K = 128; p.V = 128; p.chunk = 64;
    p.io_dtype = GDR_BF16; p.gate = GDR_GATE_SCALAR; p.scale = -1.f; p.variant = GDR_VARIANT_AUTO;
    if (gdr_version() <= 0) return 1;
    if (gdr_forward_workspace_bytes(&p) == 0 || gdr_backward_workspace_bytes(&p) == 0) return 2;
    if (gdr_varlen_forward_workspace_bytes(&p) == 0) return 3;
    if (gdr_forward(&p, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL) != GDR_ERR_NULL) return 4;
    p.K = 96;
    if (gdr_forward_workspace_bytes(&p) != 0) return 5;
    printf("%s\n", gdr_status_string(GDR_ERR_SHAPE));
    return 0;
}
""")
    libdir = os.path.dirname(gdr.LIB_PATH)
    exe = tmp_path / "use_gdr"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-L", libdir,
                    "-lgdr", "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.strip() == gdr.gdr_status_string(2)


def test_library_exports_only_the_c_abi(lib):
    # every exported function of libgdr is a gdr_* entry point the header declares; the rest of the library
    # (kernels, launchers, the CUDA runtime) stays hidden.  C++ runtime template statics (mangled _ZZ...) are
    # emitted weak by the compiler and are not part of the interface.
    import shutil
    import subprocess
    if shutil.which("nm") is None:
        pytest.skip("no nm")
    out = subprocess.run(["nm", "-D", "--defined-only", gdr.LIB_PATH], capture_output=True, text=True, check=True)
    names = [ln.split()[-1] for ln in out.stdout.splitlines() if ln.strip()]
    exported = {n for n in names if not n.startswith("_ZZ")}
    assert exported == set(declared_functions())


def test_host_forward_scratch_formula(lib):
    # two slots of one piece's q, k, v, g, beta and o ([B, T_piece, ...], each rounded up to 256 bytes),
    # three fp32 states [B, HV, K, V] (two alternating, h0), then gdr_forward's workspace for the longest
    # piece and for the last one, whichever is larger
    r = lambda x: (x + 255) // 256 * 256
    for (B, T, H, HV, K, V, C, bf16, per_k, pieces) in [(1, 32768, 32, 32, 128, 128, 64, 1, False, 8),
                                                        (2, 1000, 2, 4, 128, 128, 64, 1, False, 5),
                                                        (2, 700, 3, 3, 64, 64, 32, 0, True, 0),
                                                        (1, 100, 1, 1, 64, 64, 64, 1, False, 64)]:
        p = gdr.make_problem(B, T, H, K, V, C, 1 if bf16 else 0, per_k, HV=HV if HV != H else 0)
        e = 2 if bf16 else 4
        nt = -(-T // C)
        n = min(pieces or 8, 64, nt)
        cpp = -(-nt // n)
        Tp = min(cpp * C, T)
        last = T - (-(-nt // cpp) - 1) * cpp * C
        rows = [H * K * e, H * K * e, HV * V * e, HV * (K if per_k else 1) * 4, HV * e, HV * V * e]
        want = 2 * sum(r(B * Tp * x) for x in rows) + 3 * r(B * HV * K * V * 4)
        ws = 0
        for t in (Tp, last):
            pp = gdr.make_problem(B, t, H, K, V, C, 1 if bf16 else 0, per_k, HV=HV if HV != H else 0)
            ws = max(ws, lib.gdr_forward_workspace_bytes(ctypes.byref(pp)))
        want = r(want + ws)
        assert lib.gdr_forward_host_scratch_bytes(ctypes.byref(p), pieces) == want
    p = gdr.make_problem(1, 256, 2, 64, 64, 64, 1, False)
    assert lib.gdr_forward_host_scratch_bytes(ctypes.byref(p), -1) == 0


def test_host_forward_rejects_bad_arguments_before_launching(lib):
    p = gdr.make_problem(1, 256, 2, 64, 64, 64, 1, False)
    a = ctypes.c_void_p(16)
    args = [a] * 5
    assert lib.gdr_forward_host(ctypes.byref(p), *args, None, a, None, 0, None, 0, None) == 5   # no scratch
    assert lib.gdr_forward_host(ctypes.byref(p), *args, None, a, None, -2, a, 1 << 40, None) == 9
    assert lib.gdr_forward_host(ctypes.byref(p), None, *args[1:], None, a, None, 0, a, 1 << 40, None) == 1
    bad = gdr.make_problem(1, 256, 2, 96, 64, 64, 1, False)
    assert lib.gdr_forward_host(ctypes.byref(bad), *args, None, a, None, 0, a, 1 << 40, None) == 2


def test_fused_tc_per_key_gate_workspace(lib):
    # per-key-dim gate on the tcgen05 path: g_cum [B,T,HV,K] fp32, w, u, P [B,NT,HV,C,C], then the gated
    # operands kg and qg [B,T,HV,K] (bf16), each rounded up to 256 bytes; no pieces (one call), no segments
    r = lambda x: (x + 255) // 256 * 256
    for (B, T, H, HV) in [(2, 8192, 16, 16), (1, 100, 2, 4), (1, 32768, 4, 4)]:
        p = gdr.make_problem(B, T, H, 128, 128, 64, 1, True, variant="fused_tc", HV=HV if HV != H else 0,
                             segments=1)
        rows, nt = B * T * HV, -(-T // 64)
        want = r(rows * 128 * 4) + 2 * r(rows * 128 * 2) + r(B * nt * HV * 64 * 64 * 2) + 2 * r(rows * 128 * 2)
        assert lib.gdr_forward_workspace_bytes(ctypes.byref(p)) == want


def test_gated_operands_sizes_and_gate(lib):
    # bf16, per-key-dim gate, K = V = 128, C = 64 only
    a = ctypes.c_void_p(16)
    for (K, V, C, per_k, code) in [(128, 128, 64, False, 8), (64, 64, 64, True, 8), (128, 128, 32, True, 8)]:
        p = gdr.make_problem(1, 256, 2, K, V, C, 1, per_k)
        assert lib.gdr_gated_operands(ctypes.byref(p), a, a, a, a, a, a, None) == code
    p = gdr.make_problem(1, 256, 2, 128, 128, 64, 1, True)
    assert lib.gdr_gated_operands(ctypes.byref(p), a, None, a, a, a, a, None) == 1
