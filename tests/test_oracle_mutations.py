"""Planted mistakes: each plausible error in the oracle must make a pin fail.

A mutation is one textual change to the oracle's source (a dropped term, a
flipped sign, a wrong index, a transposed operand).  The mutated copy is built
in a temporary place (never in the tree) and the pins are re-run on it; the test
passes when at least one pin rejects the mutant.  This shows that the pins in
test_oracle_pins.py would catch such a mistake in the real oracle.
"""
import json
import os
import subprocess
import types

import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_prepare_gb300.inputs import make_inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHUNKED_SRC = os.path.join(ROOT, "oracle", "chunked.py")
NAIVE_SRC = os.path.join(ROOT, "oracle", "naive_recurrence.c")
GOLDEN = os.path.join(ROOT, "tests", "golden", "worked_examples.json")


def _inputs(per_k, K=6, V=6, T=64, seed=21):
    x = make_inputs(1, T, 2, K, V, per_k_gate=per_k, io_dtype=torch.float32, with_h0=True, seed=seed)
    d = {n: t.double().numpy() for n, t in x.tensors().items()}
    d["h0"] = d["h0"] * 20
    return d


def _golden_cases():
    with open(GOLDEN) as f:
        for ex in json.load(f)["examples"]:
            T, K, V = ex["T"], ex["K"], ex["V"]
            gf = np.log(np.array(ex["g_decay_factor"]))
            yield (dict(q=np.array(ex["q"]).reshape(1, T, 1, K), k=np.array(ex["k"]).reshape(1, T, 1, K),
                        v=np.array(ex["v"]).reshape(1, T, 1, V),
                        g=gf.reshape(1, T, 1, K) if ex["gate"] == "per_key_dim" else gf.reshape(1, T, 1),
                        beta=np.array(ex["beta"]).reshape(1, T, 1), h0=np.array(ex["h0"]).reshape(1, 1, K, V)),
                   ex["scale"], np.array(ex["o"]).reshape(1, T, 1, V), np.array(ex["h_final"]).reshape(1, 1, K, V))


# ------------------------------------------------------------ chunked (numpy) mutants

CHUNKED_MUTANTS = [
    ("k_beta without exp(G), as the prepare page's fragment writes it",
     "k_beta_g = kc * bc * np.exp(Gc)", "k_beta_g = kc * bc"),
    ("gate sign flipped inside A",
     "gate = np.exp(Gc[..., i:i + 1, :] - Gc[..., :i, :])", "gate = np.exp(Gc[..., :i, :] - Gc[..., i:i + 1, :])"),
    ("beta taken from the column instead of the row",
     "A[..., i, :i] = bc[..., i:i + 1] *", "A[..., i, :i] = bc[..., :i] *"),
    ("A transposed in the substitution",
     "A[..., i, :i], X[..., :i, :]", "A[..., :i, i], X[..., :i, :]"),
    ("identity dropped from the inverse", "row[..., i] = 1.0", "row[..., i] = 0.0"),
    ("v' sign flipped", "vp = uc[:, c] - wc[:, c] @ h", "vp = uc[:, c] + wc[:, c] @ h"),
    ("state not decayed across chunks",
     "h = np.exp(G_last)[..., None] * h + ", "h = h + "),
    ("kg gate inverted",
     "np.exp(G_last[:, :, None, :] - Gc[:, c])", "np.exp(Gc[:, c] - G_last[:, :, None, :])"),
    ("checkpoint taken after the update",
     "        ckpt[:, c] = h\n        vp = uc[:, c] - wc[:, c] @ h",
     "        vp = uc[:, c] - wc[:, c] @ h"),
    ("gate cumsum not restarted per chunk",
     "return np.cumsum(gc, axis=2).reshape(g.shape)", "return np.cumsum(g, axis=1)"),
    ("output diagonal excluded",
     "Qt[..., i, :i + 1] = np.einsum(\"...d,...jd->...j\", qc[..., i, :], kc[..., :i + 1, :] * gate)",
     "Qt[..., i, :i] = np.einsum(\"...d,...jd->...j\", qc[..., i, :], kc[..., :i, :] * gate[..., :i, :])"),
    ("scale on the inter-chunk term only",
     "scale * (inter + intra)", "scale * inter + intra"),
    ("query not gated in the inter-chunk term",
     "inter = (qc * np.exp(Gc)) @ ckpt", "inter = qc @ ckpt"),
    ("checkpoint transposed in the output",
     "inter = (qc * np.exp(Gc)) @ ckpt", "inter = (qc * np.exp(Gc)) @ np.swapaxes(ckpt, -1, -2)"),
]


def _chunked_pins_fail(mod) -> bool:
    """True when some pin rejects this version of the chunked oracle."""
    for per_k in (False, True):
        d = _inputs(per_k)
        try:
            ref = oracle.naive_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 16, 0.5)
            got = mod.forward_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 16, 0.5)
        except Exception:
            return True
        for key in ("o", "h_final", "ckpt"):
            if np.abs(got[key] - ref[key]).max() > 1e-10:
                return True
    for args, scale, o_ref, h_ref in _golden_cases():
        got = mod.forward_chunked(args["q"], args["k"], args["v"], args["g"], args["beta"], args["h0"], 2, scale)
        if np.abs(got["o"] - o_ref).max() > 1e-12 or np.abs(got["h_final"] - h_ref).max() > 1e-12:
            return True
    return False


def _load_chunked(src: str):
    mod = types.ModuleType("chunked_mutant")
    exec(compile(src, "chunked_mutant.py", "exec"), mod.__dict__)
    return mod


def test_unmutated_chunked_passes_the_pins():
    with open(CHUNKED_SRC) as f:
        assert not _chunked_pins_fail(_load_chunked(f.read()))


@pytest.mark.parametrize("what,old,new", CHUNKED_MUTANTS, ids=[m[0] for m in CHUNKED_MUTANTS])
def test_chunked_mutant_is_caught(what, old, new):
    with open(CHUNKED_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site not found: {old!r}"
    assert _chunked_pins_fail(_load_chunked(src.replace(old, new)))


# ------------------------------------------------------------ naive (C) mutants

NAIVE_MUTANTS = [
    ("delta sign flipped", "r[jj] = bt * (vt[j0 + jj] - r[jj]);", "r[jj] = bt * (vt[j0 + jj] + r[jj]);"),
    ("beta dropped", "r[jj] = bt * (vt[j0 + jj] - r[jj]);", "r[jj] = (vt[j0 + jj] - r[jj]);"),
    ("scale dropped", "for (int64_t jj = 0; jj < nj; ++jj) ot[jj] *= J->scale;", ""),
    ("per-key gate read from the first key only", "dk[i] = exp(J->g[tok * K + i]);", "dk[i] = exp(J->g[tok * K]);"),
    ("initial state transposed", "S[i * nj + jj] = src[i * V + j0 + jj];", "S[i * nj + jj] = src[(j0 + jj) * V + i];"),
    ("output read with k instead of q", "const double qi = qt[i];", "const double qi = kt[i];"),
    ("no decay", "S[i * nj + jj] *= dk[i];", "(void)dk;"),
]


def _naive_pins_fail(lib) -> bool:
    for args, scale, o_ref, h_ref in _golden_cases():
        got = oracle.naive_forward(args["q"], args["k"], args["v"], args["g"], args["beta"], args["h0"],
                                   1, scale, lib=lib)
        if np.abs(got["o"] - o_ref).max() > 1e-12 or np.abs(got["h_final"] - h_ref).max() > 1e-12:
            return True
    # square problems, so that a transposed K x V operand still has the right shape
    from test_oracle_pins import explicit_matrix_recurrence
    for per_k in (False, True):
        d = _inputs(per_k, T=16)
        o_ref, h_ref = explicit_matrix_recurrence(d, 0.5)
        got = oracle.naive_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 8, 0.5, lib=lib)
        if np.abs(got["o"] - o_ref).max() > 1e-12 or np.abs(got["h_final"] - h_ref).max() > 1e-12:
            return True
    return False


def _build_naive(src: str, tmp_path, tag: str):
    c = tmp_path / f"mut_{tag}.c"
    so = tmp_path / f"mut_{tag}.so"
    c.write_text(src)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", str(c), "-o", str(so), "-lm"])
    return oracle.load_library(str(so))


def test_unmutated_naive_passes_the_pins(tmp_path):
    with open(NAIVE_SRC) as f:
        assert not _naive_pins_fail(_build_naive(f.read(), tmp_path, "none"))


@pytest.mark.parametrize("what,old,new", NAIVE_MUTANTS, ids=[m[0] for m in NAIVE_MUTANTS])
def test_naive_mutant_is_caught(what, old, new, tmp_path):
    with open(NAIVE_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site not found: {old!r}"
    idx = NAIVE_MUTANTS.index((what, old, new))
    assert _naive_pins_fail(_build_naive(src.replace(old, new), tmp_path, str(idx)))


# ------------------------------------------------------------ backward: token reverse mode (C) mutants

ADJ_SRC = os.path.join(ROOT, "oracle", "naive_adjoint.c")
CHUNKED_BWD_SRC = os.path.join(ROOT, "oracle", "chunked_backward.py")

ADJ_MUTANTS = [
    ("read-out gradient dropped", "dS[i * V + j] += J->scale * qt[i] * dot[j];", ";"),
    ("dq read from the state before the token", "s += St[i * V + j] * dot[j];", "s += Sprev[i * V + j] * dot[j];"),
    ("dbeta taken on delta instead of r", "db += r[j] * dd[j];", "db += bt * r[j] * dd[j];"),
    ("k's path through r sign flipped", "dkt[i] -= s;", "dkt[i] += s;"),
    ("k dr^T term dropped from dS~", "dSt[i * V + j] = dS[i * V + j] - kt[i] * dr[j];",
     "dSt[i * V + j] = dS[i * V + j];"),
    ("state gradient not decayed", "dS[i * V + j] = dec[i] * dSt[i * V + j];", "dS[i * V + j] = dSt[i * V + j];"),
]


def _adjoint_pins_fail(lib) -> bool:
    from test_oracle_backward_pins import GRADS, autograd_grads, problem
    for per_k in (False, True):
        d, do, dhf = problem(per_k, B=1, T=24, seed=31)
        ref = autograd_grads(d, do, dhf, 0.45)
        got = oracle.naive_backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], do, dhf, 8, 0.45, lib=lib)
        for name in GRADS:
            if np.abs(got[name] - ref[name]).max() > 1e-10 * max(np.abs(ref[name]).max(), 1.0):
                return True
    return False


def _build_adjoint(src: str, tmp_path, tag: str):
    c = tmp_path / f"adj_{tag}.c"
    so = tmp_path / f"adj_{tag}.so"
    c.write_text(src)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", str(c), "-o", str(so), "-lm"])
    return oracle.load_adjoint_library(str(so))


def test_unmutated_adjoint_passes_the_pins(tmp_path):
    with open(ADJ_SRC) as f:
        assert not _adjoint_pins_fail(_build_adjoint(f.read(), tmp_path, "none"))


@pytest.mark.parametrize("what,old,new", ADJ_MUTANTS, ids=[m[0] for m in ADJ_MUTANTS])
def test_adjoint_mutant_is_caught(what, old, new, tmp_path):
    with open(ADJ_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site not found: {old!r}"
    assert _adjoint_pins_fail(_build_adjoint(src.replace(old, new), tmp_path, str(ADJ_MUTANTS.index((what, old, new)))))


# ------------------------------------------------------------ backward: chunked (numpy) mutants

CHUNKED_BWD_MUTANTS = [
    ("v' gradient misses the state path", "dvp = dlc[:, c] + kg @ dh", "dvp = dlc[:, c]"),
    ("reverse scan not decayed", "np.exp(G_last)[..., :, None] * dh", "dh"),
    ("output score gradient not causal", "dQt = scale * (doc @ np.swapaxes(vpc, -1, -2)) * mask",
     "dQt = scale * (doc @ np.swapaxes(vpc, -1, -2))"),
    ("kg's gate gradient sign flipped", "- kc * Rq - dkg * kg", "- kc * Rq + dkg * kg"),
    ("state decay missing from the last row's gate gradient",
     " + np.exp(G_L[..., 0, :]) * (h * dhn).sum(axis=-1)", ""),
    ("dA keeps its diagonal", "dA = np.tril(-TiT @ dT @ TiT, -1)", "dA = np.tril(-TiT @ dT @ TiT)"),
    ("beta's path through A dropped", " + (dA * M).sum(-1)", ""),
    ("padded rows' gate gradient lost", "out[:, T - 1] += dG[:, T:].sum(axis=1)", "pass"),
    ("inclusive instead of reverse cumsum",
     "out = np.flip(np.cumsum(np.flip(dc, axis=2), axis=2), axis=2).reshape(pad.shape)[:, :T]",
     "out = np.cumsum(dc, axis=2).reshape(pad.shape)[:, :T]"),
]


def _chunked_bwd_pins_fail(mod) -> bool:
    from test_oracle_backward_pins import GRADS, problem
    for per_k in (False, True):
        for T, C in ((64, 16), (100, 32)):
            d, do, dhf = problem(per_k, T=T, seed=33 + T)
            ref = oracle.naive_backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], do, dhf, C, 0.4)
            try:
                got = mod.backward_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], do, dhf, C, 0.4)
            except Exception:
                return True
            for name in GRADS:
                if np.abs(got[name] - ref[name]).max() > 1e-10 * max(np.abs(ref[name]).max(), 1.0):
                    return True
    return False


def _load_chunked_bwd(src: str):
    mod = types.ModuleType("oracle.chunked_backward_mutant")
    mod.__package__ = "oracle"
    exec(compile(src, "chunked_backward_mutant.py", "exec"), mod.__dict__)
    return mod


def test_unmutated_chunked_backward_passes_the_pins():
    with open(CHUNKED_BWD_SRC) as f:
        assert not _chunked_bwd_pins_fail(_load_chunked_bwd(f.read()))


@pytest.mark.parametrize("what,old,new", CHUNKED_BWD_MUTANTS, ids=[m[0] for m in CHUNKED_BWD_MUTANTS])
def test_chunked_backward_mutant_is_caught(what, old, new):
    with open(CHUNKED_BWD_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site not found: {old!r}"
    assert _chunked_bwd_pins_fail(_load_chunked_bwd(src.replace(old, new)))


# ------------------------------------------------------------ grouped value heads

def test_grouping_by_remainder_is_caught():
    # a value head reading q/k head hv % H (np.tile) instead of hv // G (np.repeat)
    with open(CHUNKED_SRC) as f:
        src = f.read()
    old = "return np.repeat(x, HV // H, axis=2)"
    assert src.count(old) == 1
    mod = _load_chunked(src.replace(old, "return np.tile(x, (1, 1, HV // H) + (1,) * (x.ndim - 3))"))
    from test_oracle_pins import explicit_matrix_recurrence, grouped
    d = grouped(False, H=2, G=2, seed=53)
    got = mod.forward_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], 8, 0.4)
    hv, G = 1, 2                      # value head 1 belongs to q/k head 0
    one = dict(q=d["q"][:, :, hv // G: hv // G + 1], k=d["k"][:, :, hv // G: hv // G + 1],
               v=d["v"][:, :, hv:hv + 1], g=d["g"][:, :, hv:hv + 1], beta=d["beta"][:, :, hv:hv + 1],
               h0=d["h0"][:, hv:hv + 1])
    eo, _ = explicit_matrix_recurrence(one, 0.4)
    assert np.abs(got["o"][:, :, hv:hv + 1] - eo).max() > 1e-6


# ------------------------------------------------------------ segment maps

SEGMENTS_SRC = os.path.join(ROOT, "oracle", "segments.py")

SEGMENT_MUTANTS = [
    ("chunk maps composed in the wrong order", "m = A[:, c] @ m", "m = m @ A[:, c]"),
    ("Z not carried through later chunks", "z = A[:, c] @ z + Bc[:, c]", "z = z + Bc[:, c]"),
    ("decay dropped from the chunk map", 'A = np.einsum("...d,de->...de", decay, np.eye(K)) - ',
     "A = np.eye(K) - "),
    ("kg without its gate", "kg = kc * np.exp(G_last - Gc)", "kg = kc"),
    ("segment start recorded after its update", "        starts[:, s] = h\n        h = M[:, s] @ h + Z[:, s]",
     "        h = M[:, s] @ h + Z[:, s]\n        starts[:, s] = h"),
    ("reverse stitch without the transpose", "e = np.swapaxes(M[:, s], -1, -2) @ e + Zb[:, s]", "e = M[:, s] @ e + Zb[:, s]"),
    ("reverse stitch in forward order", "for s in range(S - 1, -1, -1):", "for s in range(S):"),
]


def _segment_pins_fail(mod) -> bool:
    import test_oracle_segment_pins as pins
    checks = [lambda: pins.test_one_token_chunks_are_reflections()]
    for per_k in (False, True):
        checks.append(lambda per_k=per_k: pins.test_no_delta_step_leaves_the_decay(per_k))
        checks.append(lambda per_k=per_k: pins.test_stitched_maps_reproduce_the_serial_scan(per_k, 16, 4))
        checks.append(lambda per_k=per_k: pins.test_reverse_stitch_reproduces_the_serial_reverse_scan(per_k, 16, 4))
    saved = pins.segments
    pins.segments = mod
    try:
        for check in checks:
            try:
                check()
            except Exception:
                return True
        return False
    finally:
        pins.segments = saved


def _load_segments(src: str):
    mod = types.ModuleType("oracle.segments_mutant")
    mod.__package__ = "oracle"
    exec(compile(src, "segments_mutant.py", "exec"), mod.__dict__)
    return mod


def test_unmutated_segments_pass_the_pins():
    with open(SEGMENTS_SRC) as f:
        assert not _segment_pins_fail(_load_segments(f.read()))


@pytest.mark.parametrize("what,old,new", SEGMENT_MUTANTS, ids=[m[0] for m in SEGMENT_MUTANTS])
def test_segment_mutant_is_caught(what, old, new):
    with open(SEGMENTS_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site not found: {old!r}"
    assert _segment_pins_fail(_load_segments(src.replace(old, new)))


# ------------------------------------------------------------ packed variable-length sequences

VARLEN_SRC = os.path.join(ROOT, "oracle", "varlen.py")

VARLEN_MUTANTS = [
    ("state carried into the next sequence", '        hf[s] = r["h_final"][0]\n    return o, hf',
     '        hf[s] = r["h_final"][0]\n        if s + 1 < n:\n            h0[s + 1] = hf[s]\n    return o, hf'),
    ("an empty sequence ends in the zero state", "            hf[s] = h0[s]\n", "            hf[s] = 0.0\n"),
    ("a sequence reads the next one's first token",
     "r = naive_forward(q[None, a:b], k[None, a:b],", "r = naive_forward(q[None, a + 1:b + 1], k[None, a:b],"),
    ("outputs placed one row late", '        o[a:b] = r["o"][0]', '        o[a + 1:b + 1] = r["o"][0][:len(o[a + 1:b + 1])]'),
    ("an empty sequence drops the final-state gradient", '            out["dh0"][s] = dhf[s]',
     '            out["dh0"][s] = 0.0'),
    ("the backward reads do from the packed start", "do[None, a:b], dhf[s:s + 1]", "do[None, 0:b - a], dhf[s:s + 1]"),
]


def _varlen_pins_fail(mod) -> bool:
    import test_oracle_varlen_pins as pins
    checks = [lambda: pins.test_one_token_sequences_closed_form()]
    for per_k in (False, True):
        checks.append(lambda per_k=per_k: pins.test_equal_lengths_are_the_batch(per_k))
        checks.append(lambda per_k=per_k: pins.test_sequences_do_not_see_each_other(per_k))
        checks.append(lambda per_k=per_k: pins.test_empty_sequence_passes_its_state(per_k))
        checks.append(lambda per_k=per_k: pins.test_backward_matches_finite_differences(per_k))
    saved = pins.varlen
    pins.varlen = mod
    try:
        for check in checks:
            try:
                check()
            except Exception:
                return True
        return False
    finally:
        pins.varlen = saved


def _load_varlen(src: str):
    mod = types.ModuleType("oracle.varlen_mutant")
    mod.__package__ = "oracle"
    exec(compile(src, "varlen_mutant.py", "exec"), mod.__dict__)
    return mod


def test_unmutated_varlen_passes_the_pins():
    with open(VARLEN_SRC) as f:
        assert not _varlen_pins_fail(_load_varlen(f.read()))


@pytest.mark.parametrize("what,old,new", VARLEN_MUTANTS, ids=[m[0] for m in VARLEN_MUTANTS])
def test_varlen_mutant_is_caught(what, old, new):
    with open(VARLEN_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site not found: {old!r}"
    assert _varlen_pins_fail(_load_varlen(src.replace(old, new)))
