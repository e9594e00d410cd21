"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Every case draws seeded synthetic inputs on the GPU, runs the kernels through
``glu_quant_fwd`` / ``glu_quant_bwd``, copies inputs and outputs to the host
and checks them against ``oracle`` run on the very same input bytes, under
the rules in ``parity_util``.  Small cases span several tiles with ragged
row and column tails; the workload cases run at full size (the largest one
on sampled 32-row groups, in the launch configuration the bench times).
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from parity_util import Stats, check_mx, check_nvfp4, check_plain, host, host_bits

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import fp4_quant_gb300 as G  # noqa: E402  (raises if the library is missing)

DEV = torch.device("cuda:0")
ACTS = [(G.ACT_SILU, O.SILU), (G.ACT_GELU_TANH, O.GELU_TANH), (G.ACT_RELU, O.RELU),
        (G.ACT_IDENTITY, O.IDENTITY), (G.ACT_GELU_ERF, O.GELU_ERF)]
ACT_IDS = ["silu", "gelu", "relu", "identity", "gelu_erf"]
MODES = [G.MODE_ROW, G.MODE_COL, G.MODE_BOTH]


def _randn(M, N, seed, scale=1.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return (torch.randn(M, N, generator=g, device=DEV) * scale).to(torch.bfloat16)


def _interleave(g, u):
    M, N = g.shape
    return torch.stack([g, u], dim=-1).reshape(M, 2 * N).contiguous()


def run_fwd(g, u, act, fmt, mode, layout):
    """GPU and oracle forward on the same bytes; returns (gpu, ref) dicts."""
    if layout == G.LAYOUT_SPLIT:
        out = G.fwd(g, u, act=act, fmt=fmt, mode=mode, layout=layout)
        torch.cuda.synchronize()
        ref = O.glu_fwd(host_bits(g), host_bits(u), act=act, fmt=fmt, mode=mode,
                        layout=O.SPLIT, want_h=True)
    else:
        x = _interleave(g, u)
        out = G.fwd(x, None, act=act, fmt=fmt, mode=mode, layout=layout)
        torch.cuda.synchronize()
        ref = O.glu_fwd(host_bits(x), act=act, fmt=fmt, mode=mode, layout=O.INTERLEAVED,
                        want_h=True)
    return {k: host(v) for k, v in out.items()}, ref


def run_bwd(g, u, d, act, fmt, mode, layout):
    if layout == G.LAYOUT_SPLIT:
        out = G.bwd(g, u, d, act=act, fmt=fmt, mode=mode, layout=layout)
        torch.cuda.synchronize()
        ref = O.glu_bwd(host_bits(g), host_bits(u), host_bits(d), act=act, fmt=fmt, mode=mode,
                        layout=O.SPLIT, want_h=True)
    else:
        x = _interleave(g, u)
        out = G.bwd(x, None, d, act=act, fmt=fmt, mode=mode, layout=layout)
        torch.cuda.synchronize()
        ref = O.glu_bwd(host_bits(x), None, host_bits(d), act=act, fmt=fmt, mode=mode,
                        layout=O.INTERLEAVED, want_h=True)
    return {k: host(v) for k, v in out.items()}, ref


def check(gpu, ref, fmt, mode, M, W, what):
    st = Stats()
    if fmt == G.FMT_MXFP8:
        check_mx(gpu, ref, mode, st, what)
    elif fmt == G.FMT_NVFP4:
        check_nvfp4(gpu, ref, M, W, st, what)
    else:
        check_plain(gpu["out"], ref, fmt, st, what)
    return st


# ------------------------------------------------------------ small, ragged --

@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("mode", MODES, ids=["row", "col", "both"])
@pytest.mark.parametrize("layout", [G.LAYOUT_SPLIT, G.LAYOUT_INTERLEAVED], ids=["split", "inter"])
def test_mx_fwd_small(act, mode, layout):
    M = 200 if mode == G.MODE_ROW else 160   # ragged row tile for ROW
    N = 800                                   # 3 full 256-column tiles + 32
    g, u = _randn(M, N, 11, 2.0), _randn(M, N, 12)
    gpu, ref = run_fwd(g, u, act[0], G.FMT_MXFP8, mode, layout)
    check(gpu, ref, G.FMT_MXFP8, mode, M, N, "fwd")


@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("mode", MODES, ids=["row", "col", "both"])
@pytest.mark.parametrize("layout", [G.LAYOUT_SPLIT, G.LAYOUT_INTERLEAVED], ids=["split", "inter"])
def test_mx_bwd_small(act, mode, layout):
    M = 104 if mode == G.MODE_ROW else 96
    N = 416                                   # 3 full 128-column tiles + 32
    g, u, d = _randn(M, N, 21, 2.0), _randn(M, N, 22), _randn(M, N, 23)
    gpu, ref = run_bwd(g, u, d, act[0], G.FMT_MXFP8, mode, layout)
    check(gpu, ref, G.FMT_MXFP8, mode, M, 2 * N, "bwd")


def _relaid_to_plain(flat, R, C):
    """128x4 layout -> plain [R, C] scale matrix (padding dropped)."""
    cp = -(-C // 4) * 4
    r = np.arange(R)[:, None]
    c = np.arange(C)[None, :]
    off = ((r // 128) * (cp // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)
    return flat[off]


def check_mx_128x4(gpu, ref_plain, mode, M, W, what):
    """MXFP8 with 128x4 scales: the whole padded scale buffers equal the
    oracle's plain scales re-laid (padding zero), and the codes and scales
    pass the MXFP8 rules against the plain oracle."""
    st = Stats()
    plain = dict(gpu)
    if mode & G.MODE_ROW:
        assert np.array_equal(gpu["s_row"], O.scales_128x4(ref_plain["s_row"])), what + ".row scales"
        plain["s_row"] = _relaid_to_plain(gpu["s_row"], M, W // 32)
    if mode & G.MODE_COL:
        assert np.array_equal(gpu["s_col"], O.scales_128x4(ref_plain["s_col"])), what + ".col scales"
        plain["s_col"] = _relaid_to_plain(gpu["s_col"], W, M // 32)
    check_mx(plain, ref_plain, mode, st, what)
    return st


@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("mode", MODES, ids=["row", "col", "both"])
@pytest.mark.parametrize("direction", ["fwd", "bwd"])
def test_mx_128x4_scales(act, mode, direction):
    """MXFP8 with scales in the 128x4 layout: padded rows (M, 2N not
    multiples of 128) and padded scale columns (N/32, M/32 not multiples
    of 4); the scale buffers are filled with garbage first so that the
    padding must be written."""
    M, N = (160, 800) if direction == "fwd" else (96, 416)
    W = N if direction == "fwd" else 2 * N
    g, u, d = _randn(M, N, 41, 2.0), _randn(M, N, 42), _randn(M, N, 43)
    sizes = {"s_row": (-(-M // 128) * 128) * (-(-(W // 32) // 4) * 4),
             "s_col": (-(-W // 128) * 128) * (-(-(M // 32) // 4) * 4)}
    out = {"q_row": torch.empty((M, W), dtype=torch.uint8, device=DEV) if mode & G.MODE_ROW else None,
           "s_row": torch.full((sizes["s_row"],), 0xA5, dtype=torch.uint8, device=DEV) if mode & G.MODE_ROW else None,
           "q_col": torch.empty((W, M), dtype=torch.uint8, device=DEV) if mode & G.MODE_COL else None,
           "s_col": torch.full((sizes["s_col"],), 0xA5, dtype=torch.uint8, device=DEV) if mode & G.MODE_COL else None,
           "out": None}
    if direction == "fwd":
        G.fwd(g, u, act=act[0], fmt=G.FMT_MXFP8_128X4, mode=mode, out=out)
        ref = O.glu_fwd(host_bits(g), host_bits(u), act=act[1], fmt=O.MXFP8, mode=mode, want_h=True)
    else:
        G.bwd(g, u, d, act=act[0], fmt=G.FMT_MXFP8_128X4, mode=mode, out=out)
        ref = O.glu_bwd(host_bits(g), host_bits(u), host_bits(d), act=act[1], fmt=O.MXFP8, mode=mode,
                        want_h=True)
    torch.cuda.synchronize()
    check_mx_128x4({k: host(v) for k, v in out.items()}, ref, mode, M, W, direction)


@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("layout", [G.LAYOUT_SPLIT, G.LAYOUT_INTERLEAVED], ids=["split", "inter"])
@pytest.mark.parametrize("shape", [(200, 1296), (128, 64), (1, 16)], ids=["ragged", "one_tile", "tiny"])
def test_nvfp4_small(act, layout, shape):
    M, N = shape
    g, u = _randn(M, N, 31, 2.0), _randn(M, N, 32, 2.0)
    gpu, ref = run_fwd(g, u, act[0], G.FMT_NVFP4, G.MODE_ROW, layout)
    check(gpu, ref, G.FMT_NVFP4, G.MODE_ROW, M, N, "nvfp4")


@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("fmt", [G.FMT_BF16, G.FMT_FP32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("layout", [G.LAYOUT_SPLIT, G.LAYOUT_INTERLEAVED], ids=["split", "inter"])
@pytest.mark.parametrize("N", [1024, 1001], ids=["vec", "ragged"])
@pytest.mark.parametrize("bwd", [False, True], ids=["fwd", "bwd"])
def test_plain_small(act, fmt, layout, N, bwd):
    M = 67
    # pad the row strides to a multiple of 8 for the ragged cases (split: ld
    # >= N; interleaved: ld >= 2N)
    ld = -(-N // 8) * 8
    base_g, base_u, base_d = _randn(M, ld, 41, 2.0), _randn(M, ld, 42), _randn(M, ld, 43)
    g, u, d = base_g[:, :N], base_u[:, :N], base_d[:, :N]
    if layout == G.LAYOUT_INTERLEAVED:
        ldx = -(-2 * N // 8) * 8
        x = torch.zeros(M, ldx, dtype=torch.bfloat16, device=DEV)
        x[:, :2 * N] = _interleave(g.contiguous(), u.contiguous())
    if bwd:
        if layout == G.LAYOUT_SPLIT:
            out = G.bwd(g, u, d, act=act[0], fmt=fmt, N=N)
            torch.cuda.synchronize()
            ref = O.glu_bwd(host_bits(base_g), host_bits(base_u), host_bits(base_d), act=act[0],
                            fmt=fmt, N=N, want_h=True)
        else:
            out = G.bwd(x, None, d, act=act[0], fmt=fmt, layout=layout, N=N)
            torch.cuda.synchronize()
            ref = O.glu_bwd(host_bits(x), None, host_bits(base_d), act=act[0], fmt=fmt,
                            layout=O.INTERLEAVED, N=N, want_h=True)
    else:
        if layout == G.LAYOUT_SPLIT:
            out = G.fwd(g, u, act=act[0], fmt=fmt, N=N)
            torch.cuda.synchronize()
            ref = O.glu_fwd(host_bits(base_g), host_bits(base_u), act=act[0], fmt=fmt, N=N,
                            want_h=True)
        else:
            out = G.fwd(x, None, act=act[0], fmt=fmt, layout=layout, N=N)
            torch.cuda.synchronize()
            ref = O.glu_fwd(host_bits(x), act=act[0], fmt=fmt, layout=O.INTERLEAVED, N=N, want_h=True)
    st = Stats()
    check_plain(host(out["out"]), ref, fmt, st, "plain")


# ------------------------------------------------------------- special values --

def _special_inputs(M, N, seed):
    g, u = _randn(M, N, seed, 2.0), _randn(M, N, seed + 1)
    gv = torch.tensor([0.0, -0.0, 2.0 ** -30, -(2.0 ** -30), 2.0 ** -130, 64.0, 100.0, -64.0,
                       -100.0, -200.0, -9.0, -10.0, -11.0, -12.5, -20.0, 1e30, -1e30,
                       float("inf"), float("-inf"), float("nan"), 60.0, -60.0],
                      device=DEV).to(torch.bfloat16)
    uv = torch.tensor([0.0, -0.0, 2.0 ** -120, 1e30, -1e-30, 3.0, float("inf"), 60.0],
                      device=DEV).to(torch.bfloat16)
    gen = torch.Generator(device=DEV).manual_seed(seed + 2)
    mg = torch.randint(0, 8, (M, N), generator=gen, device=DEV) == 0
    mu = torch.randint(0, 16, (M, N), generator=gen, device=DEV) == 0
    ig = torch.randint(0, gv.numel(), (M, N), generator=gen, device=DEV)
    iu = torch.randint(0, uv.numel(), (M, N), generator=gen, device=DEV)
    g = torch.where(mg, gv[ig], g)
    u = torch.where(mu, uv[iu], u)
    # a few clean blocks so the NaN/Inf convention is not the only thing seen
    g[: M // 2, :64] = _randn(M // 2, 64, seed + 3)
    u[: M // 2, :64] = _randn(M // 2, 64, seed + 4)
    return g.contiguous(), u.contiguous()


@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("layout", [G.LAYOUT_SPLIT, G.LAYOUT_INTERLEAVED], ids=["split", "inter"])
@pytest.mark.parametrize("amax", ["tensor", 100.0, 0.75], ids=["tensor_amax", "amax_100", "amax_small"])
def test_nvfp4_global_scale(act, layout, amax):
    """NVFP4 with a global scale (glu_quant_fwd_nvfp4_gs): the amax read from
    device memory; the tensor's own amax (the spike row makes the other
    values tiny after scaling), and two smaller ones (saturating codes, and
    infinite scaled values in the spike row, which take the NaN/Inf block
    rule)."""
    M, N = 200, 1296
    g, u = _randn(M, N, 71, 2.0), _randn(M, N, 72)
    u[5, :40] = 1.0e37  # spikes: h near 1e37, so v overflows for the smaller amaxes
    if amax == "tensor":
        h = O.glu_fwd(host_bits(g), host_bits(u), act=act[1], fmt=O.FP32)["out"]
        amax = float(np.abs(h).max())
    amax_t = torch.tensor([amax], dtype=torch.float32, device=DEV)
    if layout == G.LAYOUT_SPLIT:
        out = G.fwd(g, u, act=act[0], fmt=G.FMT_NVFP4, amax=amax_t)
        ref = O.glu_fwd_nvfp4_gs(host_bits(g), host_bits(u), act=act[1], amax=amax)
    else:
        x = _interleave(g, u)
        out = G.fwd(x, None, act=act[0], fmt=G.FMT_NVFP4, layout=layout, amax=amax_t)
        ref = O.glu_fwd_nvfp4_gs(host_bits(x), act=act[1], amax=amax, layout=O.INTERLEAVED)
    torch.cuda.synchronize()
    st = Stats()
    check_nvfp4({k: host(v) for k, v in out.items()}, {"out": ref["out"], "s_nvfp4": ref["s_nvfp4"], "h": ref["v"]},
                M, N, st, "nvfp4_gs")


@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("layout", [G.LAYOUT_SPLIT, G.LAYOUT_INTERLEAVED], ids=["split", "inter"])
@pytest.mark.parametrize("shape", [(200, 416), (96, 400), (1, 16)], ids=["ragged", "half_subtile", "tiny"])
def test_nvfp4_bwd(act, layout, shape):
    """NVFP4 backward: [dGate | dUp] as packed E2M1 [M, N] with 128x4 E4M3
    scales of [M, 2N/16]; ragged rows (padding rows of the scale layout), N
    a multiple of 32 plus 16 (a half sub-tile at the end of each output)."""
    M, N = shape
    g, u, d = _randn(M, N, 101, 2.0), _randn(M, N, 102), _randn(M, N, 103)
    gpu, ref = run_bwd(g, u, d, act[0], G.FMT_NVFP4, G.MODE_ROW, layout)
    check(gpu, {"out": ref["out"], "s_nvfp4": ref["s_nvfp4"], "h": ref["h"]}, G.FMT_NVFP4,
          G.MODE_ROW, M, 2 * N, "nvfp4_bwd")


@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("fmt", [G.FMT_FP32, G.FMT_BF16, G.FMT_MXFP8, G.FMT_NVFP4],
                         ids=["fp32", "bf16", "mxfp8", "nvfp4"])
@pytest.mark.parametrize("layout", [G.LAYOUT_SPLIT, G.LAYOUT_INTERLEAVED], ids=["split", "inter"])
def test_bf16_steps_fwd(act, fmt, layout):
    """act | GLU_ACT_BF16_STEPS: the eager bf16 values RN_bf16(RN_bf16(act(g))
    * up) in every output format (MXFP8 both directions), ragged shapes."""
    M, N = (160, 800) if fmt == G.FMT_MXFP8 else (200, 1296)
    g, u = _randn(M, N, 81, 2.0), _randn(M, N, 82)
    mode = G.MODE_BOTH if fmt == G.FMT_MXFP8 else G.MODE_ROW
    gpu, ref = run_fwd(g, u, act[0] | G.ACT_BF16_STEPS, fmt, mode, layout)
    assert not np.any(ref["h"].view(np.uint32) & 0xFFFF)  # the values are bf16 values
    check(gpu, ref, fmt, mode, M, N, "bf16_steps")
    if fmt in (G.FMT_FP32, G.FMT_BF16):  # exact values: bit for bit
        assert np.array_equal(gpu["out"], ref["out"])


@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
def test_every_bf16_gate_bf16_steps(act):
    """All 65536 gate patterns through the bf16-step values (MXFP8 both and
    the BF16 output), so that every gate's bf16 rounding of act(g) is
    exercised, decided fast or exactly."""
    M, N = 256, 256
    pats = torch.arange(65536, dtype=torch.int32)
    perm = torch.randperm(65536, generator=torch.Generator().manual_seed(91))
    g = pats[perm].to(torch.int16).view(torch.bfloat16).reshape(M, N).to(DEV)
    u = _randn(M, N, 92)
    a = act[0] | G.ACT_BF16_STEPS
    gpu, ref = run_fwd(g, u, a, G.FMT_MXFP8, G.MODE_BOTH, G.LAYOUT_SPLIT)
    check(gpu, ref, G.FMT_MXFP8, G.MODE_BOTH, M, N, "all_gates_bf16_steps")
    gpu, ref = run_fwd(g, u, a, G.FMT_BF16, G.MODE_ROW, G.LAYOUT_SPLIT)
    check(gpu, ref, G.FMT_BF16, G.MODE_ROW, M, N, "all_gates_bf16_steps_out")


@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("fmt", [G.FMT_FP32, G.FMT_BF16, G.FMT_MXFP8, G.FMT_NVFP4],
                         ids=["fp32", "bf16", "mxfp8", "nvfp4"])
def test_special_values_fwd(act, fmt):
    M, N = 64, 256
    g, u = _special_inputs(M, N, 51)
    mode = G.MODE_BOTH if fmt == G.FMT_MXFP8 else G.MODE_ROW
    gpu, ref = run_fwd(g, u, act[0], fmt, mode, G.LAYOUT_SPLIT)
    check(gpu, ref, fmt, mode, M, N, "special")


@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("fmt", [G.FMT_FP32, G.FMT_MXFP8], ids=["fp32", "mxfp8"])
def test_special_values_bwd(act, fmt):
    M, N = 64, 256
    g, u = _special_inputs(M, N, 61)
    d = _randn(M, N, 63)
    d[::7, ::5] = torch.tensor(1e30, device=DEV).to(torch.bfloat16)
    d[::11, ::3] = 0.0
    mode = G.MODE_BOTH if fmt == G.FMT_MXFP8 else G.MODE_ROW
    gpu, ref = run_bwd(g, u, d, act[0], fmt, mode, G.LAYOUT_SPLIT)
    check(gpu, ref, fmt, mode, M, 2 * N, "special_bwd")


@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("direction", ["fwd", "bwd"])
def test_every_bf16_gate(act, direction):
    """All 65536 bf16 gate patterns (NaN, infinities, subnormals, the run
    where act' cancels, both ends of the fast range) through MXFP8 both
    modes; up and dY random, with a shuffle so that every block mixes
    magnitudes."""
    M, N = 256, 256
    pats = torch.arange(65536, dtype=torch.int32)
    perm = torch.randperm(65536, generator=torch.Generator().manual_seed(71))
    g = pats[perm].to(torch.int16).view(torch.bfloat16).reshape(M, N).to(DEV)
    u = _randn(M, N, 72)
    if direction == "fwd":
        gpu, ref = run_fwd(g, u, act[0], G.FMT_MXFP8, G.MODE_BOTH, G.LAYOUT_SPLIT)
        check(gpu, ref, G.FMT_MXFP8, G.MODE_BOTH, M, N, "all_gates_fwd")
    else:
        d = _randn(M, N, 73)
        gpu, ref = run_bwd(g, u, d, act[0], G.FMT_MXFP8, G.MODE_BOTH, G.LAYOUT_SPLIT)
        check(gpu, ref, G.FMT_MXFP8, G.MODE_BOTH, M, 2 * N, "all_gates_bwd")


@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("layout", [G.LAYOUT_SPLIT, G.LAYOUT_INTERLEAVED], ids=["split", "inter"])
def test_every_bf16_gate_nvfp4(act, layout):
    """All 65536 bf16 gate patterns through the NVFP4 forward (shuffled, up
    random and scaled so that blocks reach every scale and the s = 0 case)."""
    M, N = 256, 256
    pats = torch.arange(65536, dtype=torch.int32)
    perm = torch.randperm(65536, generator=torch.Generator().manual_seed(74))
    g = pats[perm].to(torch.int16).view(torch.bfloat16).reshape(M, N).to(DEV)
    u = _randn(M, N, 75)
    u[::5] *= 1e-3
    gpu, ref = run_fwd(g, u, act[0], G.FMT_NVFP4, G.MODE_ROW, layout)
    check(gpu, ref, G.FMT_NVFP4, G.MODE_ROW, M, N, "all_gates_nvfp4")


def _bits_equal(gpu, ref, fmt):
    """Every output byte equal (the NVFP4 codes and scales are "out" and
    "s_nvfp4" on the oracle's side)."""
    if fmt == G.FMT_NVFP4:
        pairs = [("q_row", "out"), ("s_row", "s_nvfp4")]
    elif fmt == G.FMT_MXFP8:
        pairs = [(k, k) for k in ("q_row", "s_row", "q_col", "s_col") if gpu.get(k) is not None]
    else:
        pairs = [("out", "out")]
    assert pairs
    for kg, kr in pairs:
        a, b = np.ascontiguousarray(gpu[kg]), np.ascontiguousarray(ref[kr])
        assert a.nbytes == b.nbytes and np.array_equal(a.reshape(-1).view(np.uint8),
                                                       b.reshape(-1).view(np.uint8)), (kg, fmt)


@pytest.mark.parametrize("act", [G.ACT_RELU, G.ACT_IDENTITY], ids=["relu", "identity"])
@pytest.mark.parametrize("steps", [0, G.ACT_BF16_STEPS], ids=["fp32", "bf16_steps"])
@pytest.mark.parametrize("layout", [G.LAYOUT_SPLIT, G.LAYOUT_INTERLEAVED], ids=["split", "inter"])
def test_exact_gates_bit_for_bit(act, steps, layout):
    """ReLU and identity gates: every value is an exact product rounded once,
    so every output byte (codes, scales, signed zeros, fp32/bf16 bits)
    equals the oracle's, with no tolerance window; ragged shapes, +-0 and
    spiked operands, forward (every format) and backward (MXFP8 row, col,
    both; NVFP4; FP32)."""
    M, N = 160, 800
    g, u, d = _randn(M, N, 301, 2.0), _randn(M, N, 302), _randn(M, N, 303)
    g[::9, ::4] = 0.0
    g[::13, 1::4] = -0.0
    u[::7, ::6] = -0.0
    g[::31, ::17] = 60.0
    d[::5, ::11] = 0.0
    a = act | steps
    for fmt, mode in ((G.FMT_MXFP8, G.MODE_BOTH), (G.FMT_NVFP4, G.MODE_ROW), (G.FMT_FP32, G.MODE_ROW),
                      (G.FMT_BF16, G.MODE_ROW)):
        gpu, ref = run_fwd(g, u, a, fmt, mode, layout)
        _bits_equal(gpu, ref, fmt)
    if steps:
        return
    for fmt, mode in ((G.FMT_MXFP8, G.MODE_ROW), (G.FMT_MXFP8, G.MODE_COL), (G.FMT_MXFP8, G.MODE_BOTH),
                      (G.FMT_NVFP4, G.MODE_ROW), (G.FMT_FP32, G.MODE_ROW)):
        gpu, ref = run_bwd(g, u, d, act, fmt, mode, layout)
        _bits_equal(gpu, ref, fmt)


def test_exact_activation_blocks_on_gpu():
    # gate = 32: h = 32 * up exactly; amax at 448 * 2^k, ties, subnormal codes
    M, N = 32, 64
    up = torch.zeros(M, N)
    up[:, 0] = 14.0
    up[:, 1] = 2.0 ** -14
    up[:, 2] = 3 * 2.0 ** -15
    up[:, 3] = 17 * 2.0 ** -9
    up[:, 4] = -(2.0 ** -16)
    up[:, 32] = 28.0
    g = torch.full((M, N), 32.0, device=DEV).to(torch.bfloat16)
    u = up.to(DEV).to(torch.bfloat16)
    for act in (G.ACT_SILU, G.ACT_GELU_TANH):
        gpu, ref = run_fwd(g, u, act, G.FMT_MXFP8, G.MODE_BOTH, G.LAYOUT_SPLIT)
        assert list(gpu["s_row"][0]) == [127, 128]
        assert list(gpu["q_row"][0, :5]) == [0x7E, 0x01, 0x02, 0x38, 0x80]
        check(gpu, ref, G.FMT_MXFP8, G.MODE_BOTH, M, N, "exact")


def test_nvfp4_codes_near_midpoints():
    # gate = 32 makes h = 32 * up exactly; with amax = 6 the scale is 1.0 and
    # v = h, so up values on and next to the E2M1 midpoints probe rounding
    M, N = 128, 64
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    vals = []
    for m in mids:
        for k in (-2, -1, 0, 1, 2):
            vals.append(m * (1 + k * 2.0 ** -7))  # neighbours on the bf16 grid
    row = torch.zeros(N)
    row[0] = 6.0
    row[1: 1 + len(vals)] = torch.tensor(vals)
    h = row.repeat(M, 1)
    h[1::2] = -h[1::2]
    g = torch.full((M, N), 32.0, device=DEV).to(torch.bfloat16)
    u = (h / 32).to(DEV).to(torch.bfloat16)
    for layout in (G.LAYOUT_SPLIT, G.LAYOUT_INTERLEAVED):
        gpu, ref = run_fwd(g, u, G.ACT_SILU, G.FMT_NVFP4, G.MODE_ROW, layout)
        st = check(gpu, ref, G.FMT_NVFP4, G.MODE_ROW, M, N, "mid")
        assert np.array_equal(gpu["q_row"], ref["out"])
        assert st.get("mid.codes.window_mismatch", 0) == 0


# ---------------------------------------------------------------- workloads --

def test_workload_swiglu_128():
    sp = synth.spec("swiglu_128")
    x = synth.make(sp, DEV)
    gpu, ref = run_fwd(x["gate"], x["up"], G.ACT_SILU, G.FMT_MXFP8, G.MODE_ROW, G.LAYOUT_SPLIT)
    assert gpu["q_row"].shape == (128, 128) and gpu["s_row"].shape == (128, 4)
    check(gpu, ref, G.FMT_MXFP8, G.MODE_ROW, 128, 128, "swiglu_128")


@pytest.fixture(scope="module")
def swiglu_4096():
    return synth.make(synth.spec("swiglu_4096"), DEV, with_dy=True)


@pytest.mark.parametrize("mode", MODES, ids=["row", "col", "both"])
@pytest.mark.parametrize("direction", ["fwd", "bwd"])
def test_workload_swiglu_4096(swiglu_4096, mode, direction):
    x = swiglu_4096
    if direction == "fwd":
        gpu, ref = run_fwd(x["gate"], x["up"], G.ACT_SILU, G.FMT_MXFP8, mode, G.LAYOUT_SPLIT)
        check(gpu, ref, G.FMT_MXFP8, mode, 4096, 7168, "swiglu_4096")
    else:
        gpu, ref = run_bwd(x["gate"], x["up"], x["dy"], G.ACT_SILU, G.FMT_MXFP8, mode,
                           G.LAYOUT_SPLIT)
        check(gpu, ref, G.FMT_MXFP8, mode, 4096, 2 * 7168, "swiglu_4096_bwd")


@pytest.mark.parametrize("N", [11008, 14336, 18944, 29568])
@pytest.mark.parametrize("fmt", [G.FMT_MXFP8, G.FMT_BF16], ids=["mxfp8", "bf16"])
@pytest.mark.parametrize("direction", ["fwd", "bwd"])
def test_workload_geglu_8192(N, fmt, direction):
    x = synth.make(synth.spec("geglu_8192", N=N), DEV, with_dy=True)
    if direction == "fwd":
        gpu, ref = run_fwd(x["gate"], x["up"], G.ACT_GELU_TANH, fmt, G.MODE_ROW, G.LAYOUT_SPLIT)
        check(gpu, ref, fmt, G.MODE_ROW, 8192, N, "geglu_8192")
    else:
        gpu, ref = run_bwd(x["gate"], x["up"], x["dy"], G.ACT_GELU_TANH, fmt, G.MODE_ROW,
                           G.LAYOUT_SPLIT)
        check(gpu, ref, fmt, G.MODE_ROW, 8192, 2 * N, "geglu_8192_bwd")


@pytest.mark.parametrize("M", [784, 968])
def test_workload_geglu_nvfp4(M):
    sp = synth.spec("geglu_nvfp4", M=M)
    x = synth.make(sp, DEV)["x"]
    out = G.fwd(x, None, act=G.ACT_GELU_TANH, fmt=G.FMT_NVFP4, layout=G.LAYOUT_INTERLEAVED)
    torch.cuda.synchronize()
    gpu = {k: host(v) for k, v in out.items()}
    assert gpu["q_row"].shape == (M, 8192)
    assert gpu["s_row"].size == (-(-M // 128) * 128) * 1024
    ref = O.glu_fwd(host_bits(x), act=O.GELU_TANH, fmt=O.NVFP4, layout=O.INTERLEAVED,
                    want_h=True)
    check(gpu, ref, G.FMT_NVFP4, G.MODE_ROW, M, 16384, "geglu_nvfp4")


@pytest.fixture(scope="module")
def swiglu_131072():
    return synth.make(synth.spec("swiglu_131072"), DEV, with_dy=True)


def _sample_groups(M, n=24):
    groups = sorted(set([0, M // 32 - 1] + list(np.linspace(1, M // 32 - 2, n).astype(int))))
    return [int(g) * 32 for g in groups]


@pytest.mark.parametrize("mode", MODES, ids=["row", "col", "both"])
@pytest.mark.parametrize("direction", ["fwd", "bwd"])
def test_workload_swiglu_131072_sampled(swiglu_131072, mode, direction):
    """Full-size launch; the oracle checks sampled 32-row groups (every
    output block of those rows, rowwise and colwise)."""
    x = swiglu_131072
    M, N = x["gate"].shape
    W = N if direction == "fwd" else 2 * N
    if direction == "fwd":
        out = G.fwd(x["gate"], x["up"], act=G.ACT_SILU, fmt=G.FMT_MXFP8, mode=mode)
    else:
        out = G.bwd(x["gate"], x["up"], x["dy"], act=G.ACT_SILU, fmt=G.FMT_MXFP8, mode=mode)
    torch.cuda.synchronize()
    st = Stats()
    for r0 in _sample_groups(M):
        sl = slice(r0, r0 + 32)
        if direction == "fwd":
            ref = O.glu_fwd(host_bits(x["gate"][sl]), host_bits(x["up"][sl]), act=O.SILU,
                            fmt=O.MXFP8, mode=mode, want_h=True)
        else:
            ref = O.glu_bwd(host_bits(x["gate"][sl]), host_bits(x["up"][sl]),
                            host_bits(x["dy"][sl]), act=O.SILU, fmt=O.MXFP8, mode=mode,
                            want_h=True)
        gpu = {}
        if mode & G.MODE_ROW:
            gpu["q_row"] = host(out["q_row"][sl])
            gpu["s_row"] = host(out["s_row"][sl])
        if mode & G.MODE_COL:
            gpu["q_col"] = host(out["q_col"][:, sl])
            gpu["s_col"] = host(out["s_col"][:, r0 // 32: r0 // 32 + 1])
        check_mx(gpu, ref, mode, st, "swiglu_131072")
    assert st["swiglu_131072." + ("row" if mode & G.MODE_ROW else "col") + ".elements"] > 0


# -------------------------------------------------- host-visible behaviour --

def test_rejected_call_writes_nothing():
    g, u = _randn(64, 256, 71), _randn(64, 256, 72)
    q = torch.full((64, 256), 0xAB, dtype=torch.uint8, device=DEV)
    s = torch.full((64, 8), 0xAB, dtype=torch.uint8, device=DEV)
    a = G.GluQuantFwdArgs(G.ACT_SILU, G.FMT_MXFP8, G.MODE_ROW, G.LAYOUT_SPLIT, 64, 256, 256,
                          g.data_ptr() + 2, u.data_ptr(), q.data_ptr(), s.data_ptr(), None, None,
                          None)
    assert G.glu_quant_fwd(a, torch.cuda.current_stream().cuda_stream) == G.GLU_EALIGN
    a.gate = g.data_ptr()
    a.N = 240
    assert G.glu_quant_fwd(a, torch.cuda.current_stream().cuda_stream) == G.GLU_ESHAPE
    torch.cuda.synchronize()
    assert bool((q == 0xAB).all()) and bool((s == 0xAB).all())


def test_repeat_calls_and_graph_replay_are_identical():
    g, u, d = _randn(512, 2048, 81), _randn(512, 2048, 82), _randn(512, 2048, 83)
    a = G.fwd(g, u, mode=G.MODE_BOTH)
    b = G.bwd(g, u, d, mode=G.MODE_BOTH)
    a2 = G.fwd(g, u, mode=G.MODE_BOTH)
    outs = {k: torch.empty_like(v) for k, v in a.items() if v is not None}
    outs.update({k: None for k, v in a.items() if v is None})
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        G.fwd(g, u, mode=G.MODE_BOTH, out=outs, stream=s.cuda_stream)  # warm-up on side stream
        with torch.cuda.graph(graph, stream=s):
            G.fwd(g, u, mode=G.MODE_BOTH, out=outs, stream=s.cuda_stream)
    for v in outs.values():
        if v is not None:
            v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for k in ("q_row", "s_row", "q_col", "s_col"):
        assert torch.equal(a[k], a2[k]) and torch.equal(a[k], outs[k]), k
    b2 = G.bwd(g, u, d, mode=G.MODE_BOTH)
    for k in ("q_row", "s_row", "q_col", "s_col"):
        assert torch.equal(b[k], b2[k])


def test_row_chunks_equal_full_batch():
    # batch invariance: each 32-row group depends on its own rows only
    g, u, d = _randn(256, 1024, 91), _randn(256, 1024, 92), _randn(256, 1024, 93)
    full = G.bwd(g, u, d, mode=G.MODE_BOTH)
    top = G.bwd(g[:96], u[:96], d[:96], mode=G.MODE_BOTH)
    bot = G.bwd(g[96:], u[96:], d[96:], mode=G.MODE_BOTH)
    assert torch.equal(full["q_row"], torch.cat([top["q_row"], bot["q_row"]]))
    assert torch.equal(full["q_col"], torch.cat([top["q_col"], bot["q_col"]], dim=1))
    assert torch.equal(full["s_col"], torch.cat([top["s_col"], bot["s_col"]], dim=1))


def test_packed_gate_up_layout():
    # [gate | up] packed in one [M, 2N] tensor: up = gate + N, ld = 2N
    M, N = 128, 512
    gu = _randn(M, 2 * N, 101)
    g, u = gu[:, :N], gu[:, N:]
    a = G.fwd(g, u, mode=G.MODE_BOTH)
    b = G.fwd(g.contiguous(), u.contiguous(), mode=G.MODE_BOTH)
    for k in ("q_row", "s_row", "q_col", "s_col"):
        assert torch.equal(a[k], b[k])


def test_device_error_bits_stay_clear():
    """No bounded wait gave up during the calls above or a fresh set of
    calls of every MXFP8 mode (the bits are read back and cleared)."""
    st, f, b = G.glu_quant_device_errors(clear=True)
    assert st == G.GLU_OK
    g, u, d = _randn(256, 512, 81), _randn(256, 512, 82), _randn(256, 512, 83)
    for mode in MODES:
        G.fwd(g, u, mode=mode)
        G.bwd(g, u, d, mode=mode)
    torch.cuda.synchronize()
    st, f, b = G.glu_quant_device_errors(clear=True)
    assert (st, f, b) == (G.GLU_OK, 0, 0)


@pytest.mark.parametrize("shape", [(128, 416), (96, 384), (256, 1024), (160, 640)],
                         ids=["units_ragged_strip", "tiles_full_strips", "units_full_strips", "ragged_unit"])
@pytest.mark.parametrize("fmt", [G.FMT_MXFP8, G.FMT_MXFP8_128X4], ids=["rowmajor", "128x4"])
@pytest.mark.parametrize("direction", ["fwd", "bwd"])
def test_scale_word_paths(shape, fmt, direction):
    """Every combination of the four-byte scale stores and their byte
    fallbacks: row tiles in whole units of four or not (colwise words), whole
    128-column strips or a ragged last strip (rowwise words across a group's
    warps), in both scale layouts, for the colwise and both-direction calls."""
    M, N = shape
    g, u, d = _randn(M, N, 111, 2.0), _randn(M, N, 112), _randn(M, N, 113)
    W = N if direction == "fwd" else 2 * N
    for mode in (G.MODE_COL, G.MODE_BOTH):
        if direction == "fwd":
            out = G.fwd(g, u, fmt=fmt, mode=mode)
            torch.cuda.synchronize()
            ref = O.glu_fwd(host_bits(g), host_bits(u), act=O.SILU, fmt=O.MXFP8, mode=mode, want_h=True)
        else:
            out = G.bwd(g, u, d, fmt=fmt, mode=mode)
            torch.cuda.synchronize()
            ref = O.glu_bwd(host_bits(g), host_bits(u), host_bits(d), act=O.SILU, fmt=O.MXFP8, mode=mode,
                            want_h=True)
        gpu = {k: host(v) for k, v in out.items()}
        if fmt == G.FMT_MXFP8:
            check(gpu, ref, G.FMT_MXFP8, mode, M, W, f"{direction}_{mode}")
        else:
            check_mx_128x4(gpu, ref, mode, M, W, f"{direction}_{mode}_128x4")
