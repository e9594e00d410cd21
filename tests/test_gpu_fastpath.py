"""The kernels' fast fp32 activation forms, measured over every bf16 gate
against the oracle's exact values: the worst relative error plus the
roundings that follow must stay inside the rounding-test half-widths the
kernels use (Bracket<ACT> in glu_common.cuh), or the rounding test could
accept a wrong code.  Units: 2^-24."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp4_quant_gb300", "csrc")

# half-widths (units of 2^-24) and measured-form ranges, per activation
BRACKET = {0: {"act": 16.0, "dup": 16.0},
           1: {"act": 64.0, "dup": 64.0},
           4: {"act": 16.0, "dup": 16.0}}
FWD_RANGE = {0: (-64.0, 64.0), 1: (-7.0, 64.0), 4: (-13.0, 64.0)}
BWD_RANGE = {0: (-64.0, 64.0), 1: (-6.0, 64.0), 4: (-13.0, 64.0)}
# the last (widest) step of the dGate ladder: 2^-14 (tables), 2^-11 (GELU erf)
WIDEST_STEP = {0: 2.0 ** -14, 1: 2.0 ** -14, 4: 2.0 ** -11}
SLACK = 1.5  # final product rounding, exact-value rounding, bracket product


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp4_quant_gb300.build as B
    B.build()  # generated tables
    out = str(tmp_path_factory.mktemp("probe") / "libprobe.so")
    subprocess.run([B._nvcc(), *B.ARCH, *B.NVCC_FLAGS, "-I", CSRC, "-I", B.INCLUDE, "-shared",
                    os.path.join(ROOT, "tests", "fastpath_probe.cu"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.gq_probe_fast.argtypes = [ctypes.c_int, ctypes.c_void_p]
    lib.gq_probe_gemm.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    res = {"lib": lib}
    for act in (0, 1, 4):
        h = np.zeros(4 * 65536, np.float32)
        assert lib.gq_probe_fast(act, h.ctypes.data) == 0
        res[act] = h.reshape(65536, 4)
    return res


def _gates():
    pats = np.arange(65536, dtype=np.uint32)
    g = (pats << 16).view(np.float32).astype(np.float64)
    return pats, g


def _max_ulps(fast, exact, sel):
    err = np.abs(fast[sel].astype(np.float64) - exact[sel]) / np.abs(exact[sel])
    return float(err.max() * 2.0 ** 24)


@pytest.mark.parametrize("act", [0, 1, 4], ids=["silu", "gelu", "gelu_erf"])
def test_forward_form(probe, act):
    h = probe[act]
    pats, g = _gates()
    lo, hi = FWD_RANGE[act]
    with np.errstate(all="ignore"):
        sel = np.isfinite(g) & (g > lo) & (g < hi) & (np.abs(g) >= 2.0 ** -126)
        ex = O.act(act, g)
        u = _max_ulps(h[:, 0], ex, sel)
    print(f"forward act max error {u:.2f} units")
    assert u + SLACK <= BRACKET[act]["act"]


def _dgate_bracket_units(n, widest):
    """The kernels' dGate half-width (dgate_bracket, dgate_bracket_erf in
    glu_common.cuh) from |N| (GELU erf: the cancellation ratio n), in units
    of 2^-24: 2^-18 for |N| >= 1/8, doubling at each halving of |N| down to
    the widest step."""
    n = np.abs(n.astype(np.float64))
    top = widest * 2.0 ** 24
    d = np.full(n.shape, top)
    e, lim = 6, 2.0 ** -3
    while 2.0 ** e < top:
        d = np.where((n >= lim) & (d == top), 2.0 ** e, d)
        e, lim = e + 1, lim / 2
    return d


@pytest.mark.parametrize("act", [0, 1, 4], ids=["silu", "gelu", "gelu_erf"])
def test_backward_forms(probe, act):
    h = probe[act]
    pats, g = _gates()
    lo, hi = BWD_RANGE[act]
    with np.errstate(all="ignore"):
        sel = np.isfinite(g) & (g > lo) & (g < hi) & (np.abs(g) >= 2.0 ** -126)
        u_up = _max_ulps(h[:, 2], O.act(act, g), sel)
        ex = O.act_grad(act, g)
        err = np.abs(h[:, 1].astype(np.float64) - ex) / np.abs(ex) * 2.0 ** 24
        # each gate's dGate error against the half-width its |N| selects
        room = _dgate_bracket_units(h[:, 3], WIDEST_STEP[act]) - (err + SLACK)
        worst = int(np.argmin(np.where(sel, room, np.inf)))
        u_gate = float(err[sel].max())
        # away from the zero of act' the closed form keeps the error of E
        # unmagnified
        far = sel & (np.abs(h[:, 3]) >= 2.0 ** -3)
        u_far = float(err[far].max())
    print(f"dUp max error {u_up:.2f}; dGate max error {u_gate:.2f} units, {u_far:.2f} where |N| >= 1/8; "
          f"least room {room[worst]:.1f} units at g = {g[worst]}")
    assert u_up + SLACK <= BRACKET[act]["dup"]
    assert room[worst] >= 0.0
    assert u_gate + SLACK <= WIDEST_STEP[act] * 2.0 ** 24
    assert u_far + SLACK <= 64.0


# The gate/up GEMM's epilogue takes fp32 gates (the accumulators): its
# forms' half-width (GemmBracket in gemm_glu.cu), units of 2^-24, and the
# fast range (gates at or below the lower end take the exact path).
GEMM_BRACKET = {0: 16.0, 1: 16.0, 4: 16.0}
GEMM_RANGE = {0: (-64.0, 64.0), 1: (-7.0, 64.0), 4: (-13.0, 64.0)}


def _f32_gates(lo, hi):
    """fp32 gates: N(0, s) for a few spreads, uniform over the range, and
    every fp32 of a few narrow windows (the tails, around 0 and +-1)."""
    rng = np.random.default_rng(2024)
    parts = [rng.standard_normal(1 << 20) * s for s in (0.5, 1.5, 4.0)]
    parts.append(rng.uniform(lo, hi, 1 << 21))
    for c in (lo + 0.5, -1.0, -2.0 ** -10, 2.0 ** -10, 1.0, 8.0):
        b = np.float32(c).view(np.uint32)
        parts.append((np.arange(-(1 << 16), 1 << 16, dtype=np.int64) + int(b)).astype(np.uint32).view(np.float32))
    g = np.concatenate([np.asarray(p, np.float32) for p in parts])
    return g[(g > lo) & (g < hi) & (np.abs(g) >= 2.0 ** -126)]


@pytest.mark.parametrize("act", [0, 1, 4], ids=["silu", "gelu", "gelu_erf"])
def test_gemm_epilogue_form(probe, act):
    """The GEMM epilogue's act(g) for fp32 gates (exponent in two words):
    worst error plus the roundings after it (the product with up, which
    for fp32 operands is one more rounding) within its half-width."""
    lo, hi = GEMM_RANGE[act]
    g = np.ascontiguousarray(_f32_gates(lo, hi))
    out = np.zeros_like(g)
    assert probe["lib"].gq_probe_gemm(act, g.ctypes.data, out.ctypes.data, g.size) == 0
    ex = O.act(act, g.astype(np.float64))
    sel = ex != 0
    u = _max_ulps(out, ex, sel)
    print(f"GEMM epilogue form max error {u:.2f} units over {g.size} gates")
    assert u + SLACK + 1.0 <= GEMM_BRACKET[act]
