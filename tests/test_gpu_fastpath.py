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
BRACKET = {0: {"act": 16.0, "dup": 16.0, "dgate": 64.0},
           1: {"act": 64.0, "dup": 64.0, "dgate": 64.0}}
FWD_RANGE = {0: (-64.0, 64.0), 1: (-7.0, 64.0)}
BWD_RANGE = {0: (-64.0, 64.0), 1: (-6.0, 64.0)}
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
    lib.gq_probe_fast.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    res = {}
    for act in (0, 1):
        h = np.zeros(4 * 65536, np.float32)
        cancel = np.zeros(2, np.uint32)
        assert lib.gq_probe_fast(act, h.ctypes.data, cancel.ctypes.data) == 0
        res[act] = (h.reshape(65536, 4), int(cancel[0]), int(cancel[1]))
    return res


def _gates():
    pats = np.arange(65536, dtype=np.uint32)
    g = (pats << 16).view(np.float32).astype(np.float64)
    return pats, g


def _max_ulps(fast, exact, sel):
    err = np.abs(fast[sel].astype(np.float64) - exact[sel]) / np.abs(exact[sel])
    return float(err.max() * 2.0 ** 24)


@pytest.mark.parametrize("act", [0, 1], ids=["silu", "gelu"])
def test_forward_form(probe, act):
    h, _, _ = probe[act]
    pats, g = _gates()
    lo, hi = FWD_RANGE[act]
    with np.errstate(all="ignore"):
        sel = np.isfinite(g) & (g > lo) & (g < hi) & (np.abs(g) >= 2.0 ** -126)
        ex = O.act(act, g)
        u = _max_ulps(h[:, 0], ex, sel)
    print(f"forward act max error {u:.2f} units")
    assert u + SLACK <= BRACKET[act]["act"]


@pytest.mark.parametrize("act", [0, 1], ids=["silu", "gelu"])
def test_backward_forms(probe, act):
    h, p0, span = probe[act]
    pats, g = _gates()
    lo, hi = BWD_RANGE[act]
    with np.errstate(all="ignore"):
        sel = np.isfinite(g) & (g > lo) & (g < hi) & (np.abs(g) >= 2.0 ** -126)
        u_up = _max_ulps(h[:, 2], O.act(act, g), sel)
        run = (pats >= p0) & (pats < p0 + span)
        u_gate = _max_ulps(h[:, 1], O.act_grad(act, g), sel & ~run)
    print(f"dUp max error {u_up:.2f}, dGate max error {u_gate:.2f} units (run {p0:#x}+{span})")
    assert u_up + SLACK <= BRACKET[act]["dup"]
    assert u_gate + SLACK <= BRACKET[act]["dgate"]
    # the run is where the fast dGate form cancels: it must be short and
    # sit around the zero of act'
    assert 1 <= span <= 16  # (the kernel copies at most 16 entries)
    assert np.all(np.abs(O.act_grad(act, g[run])) < 0.05)
