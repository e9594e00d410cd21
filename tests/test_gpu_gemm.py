"""Parity of the gate/up GEMM with the quantiser in its epilogue (through the
C ABI) with the oracle.

"feat(phyai-kernel): add Thor NVFP4 GeGLU kernel for pi0.5", Summary and
Supported contract: the merged gate/up projection (pairwise-interleaved
weight rows), the GeGLU fold and the NVFP4 store in one kernel.  Here the
operands are bf16 and the projection runs on the tcgen05 tensor cores.

Two kinds of cases:
  * operands with few significant bits (multiples of 1/4 and 1/8 below 4),
    for which every partial sum of the projection is exact in fp32, so the
    tensor cores' accumulation equals the oracle's whatever its order: codes
    and scales must then follow the usual rules exactly (scales bit-exact,
    codes bit-exact outside the 2-ulp window);
  * N(0,1) operands at the pages' shapes (M = 968, K = 2048, H = 16384,
    sampled row tiles): the fp32 accumulation differs from the oracle's
    correctly rounded sums by far less than a code step, so a code or scale
    may differ only next to a rounding boundary, by one step, and rarely.
"""
import numpy as np
import pytest
import torch

import oracle as O
from parity_util import Stats, check_codes, check_scales, host

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import fp4_quant_gb300 as G  # noqa: E402

DEV = torch.device("cuda:0")
ACTS = [(G.ACT_SILU, O.SILU), (G.ACT_GELU_TANH, O.GELU_TANH), (G.ACT_RELU, O.RELU),
        (G.ACT_IDENTITY, O.IDENTITY), (G.ACT_GELU_ERF, O.GELU_ERF)]
ACT_IDS = ["silu", "gelu", "relu", "identity", "gelu_erf"]
FMTS = [(G.FMT_NVFP4, O.NVFP4), (G.FMT_MXFP8, O.MXFP8), (G.FMT_MXFP8_128X4, O.MXFP8_128X4)]
FMT_IDS = ["nvfp4", "mxfp8", "mxfp8_128x4"]
LAYOUTS = [(G.LAYOUT_INTERLEAVED, O.INTERLEAVED), (G.LAYOUT_SPLIT, O.SPLIT)]


def _exact_operands(M, H, K, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randint(-3, 4, (M, K), generator=g).float() / 4
    w = torch.randint(-3, 4, (2 * H, K), generator=g).float() / 8
    return x.to(torch.bfloat16).to(DEV), w.to(torch.bfloat16).to(DEV)


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _unpack_nv(q, M, H):
    q = q.reshape(M, H // 2)
    return np.stack([q & 0xF, q >> 4], axis=-1).reshape(M, H)


def _mx_v(h, s_plain):
    e = np.repeat(s_plain.astype(np.int32), 32, axis=1) - 127
    return (h.astype(np.float64) * np.exp2(-e)).astype(np.float32)


def _unswizzle(s_flat, R, C):
    cp = -(-C // 4) * 4
    r = np.arange(R)[:, None]
    c = np.arange(C)[None, :]
    return s_flat[((r // 128) * (cp // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)]


def _check(gpu, ref, fmt, M, H, st, what):
    if fmt == G.FMT_NVFP4:
        check_scales(gpu["s"], ref["s"], st, what + ".scales")
        s = O.e4m3_decode(_unswizzle(ref["s"], M, H // 16)).astype(np.float32)
        sv = np.repeat(s, 16, axis=1)
        with np.errstate(divide="ignore", invalid="ignore"):
            v = np.where(sv == 0, 0, ref["h"] / np.where(sv == 0, 1, sv)).astype(np.float32)
        check_codes(_unpack_nv(gpu["q"][: M * H // 2], M, H), _unpack_nv(ref["q"], M, H), v, O.NVFP4, st,
                    what + ".codes")
    else:
        check_scales(gpu["s"], ref["s"].reshape(-1), st, what + ".scales")
        plain = ref["s"].reshape(M, H // 32) if fmt == G.FMT_MXFP8 else _unswizzle(ref["s"], M, H // 32)
        check_codes(gpu["q"][: M * H].reshape(M, H), ref["q"].reshape(M, H), _mx_v(ref["h"], plain), O.MXFP8,
                    st, what + ".codes")


def run(x, w, act, fmt, layout):
    out = G.gemm(x, w, act=act[0], fmt=fmt[0], layout=layout[0])
    torch.cuda.synchronize()
    ref = O.gemm_glu_fwd(_bits(x), _bits(w), act=act[1], fmt=fmt[1], layout=layout[1], want_h=True)
    return {k: host(v) for k, v in out.items()}, ref


@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
@pytest.mark.parametrize("layout", LAYOUTS, ids=["inter", "split"])
@pytest.mark.parametrize("shape", [(128, 128, 64), (200, 384, 256)], ids=["one_tile", "ragged"])
def test_gemm_exact_operands(act, fmt, layout, shape):
    M, H, K = shape
    x, w = _exact_operands(M, H, K, 7)
    gpu, ref = run(x, w, act, fmt, layout)
    st = Stats()
    _check(gpu, ref, fmt[0], M, H, st, "gemm")


@pytest.mark.parametrize("case", [(ACTS[1], FMTS[0], LAYOUTS[0]), (ACTS[0], FMTS[1], LAYOUTS[1]),
                                  (ACTS[4], FMTS[2], LAYOUTS[0])], ids=["geglu_nvfp4_inter", "swiglu_mxfp8_split",
                                                                      "gelu_erf_128x4_inter"])
def test_gemm_exact_operands_pages_depth(case):
    # K = 2048 (the pages' depth), several row and column tiles, a ragged
    # last row tile (968 = 7 * 128 + 72)
    act, fmt, layout = case
    M, H, K = 968, 1024, 2048
    x, w = _exact_operands(M, H, K, 8)
    gpu, ref = run(x, w, act, fmt, layout)
    st = Stats()
    _check(gpu, ref, fmt[0], M, H, st, "gemm")


def test_gemm_pages_shape_random_operands():
    """M = 968, K = 2048, H = 16384 (the pages' largest pi0.5 shape), N(0,1)
    bf16 operands, GeGLU (tanh), NVFP4, interleaved rows.  The oracle runs on
    two row tiles (the first and the ragged last one); codes and scales there
    agree with the oracle's except next to a rounding boundary, where the
    tensor cores' fp32 accumulation order may move a value across it: such
    differences are one step, and rare."""
    M, H, K = 968, 16384, 2048
    g = torch.Generator(device=DEV).manual_seed(11)
    x = torch.randn(M, K, generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn(2 * H, K, generator=g, device=DEV) / 32).to(torch.bfloat16)
    out = G.gemm(x, w, act=G.ACT_GELU_TANH, fmt=G.FMT_NVFP4, layout=G.LAYOUT_INTERLEAVED)
    torch.cuda.synchronize()
    q = host(out["q"]).reshape(M, H // 2)
    s = host(out["s"])
    xb, wb = _bits(x), _bits(w)
    for r0, r1 in ((0, 128), (896, 968)):
        ref = O.gemm_glu_fwd(xb[r0:r1], wb, act=O.GELU_TANH, fmt=O.NVFP4, layout=O.INTERLEAVED)
        n = r1 - r0
        # this row tile's 128x4 scale tiles: bytes of row tile r0 / 128
        cols = H // 16
        tile = s[(r0 // 128) * 128 * cols:(r0 // 128 + 1) * 128 * cols]
        s_gpu = _unswizzle(tile, 128, cols)[:n]
        s_ref = _unswizzle(ref["s"], 128, cols)[:n]
        bad_s = s_gpu != s_ref
        assert bad_s.mean() < 1e-3, f"rows {r0}..{r1}: {bad_s.sum()} scale differences"
        if bad_s.any():
            assert np.all(np.abs(s_gpu[bad_s].astype(int) - s_ref[bad_s].astype(int)) == 1)
        cg, cr = _unpack_nv(q[r0:r1], n, H), _unpack_nv(ref["q"], n, H)
        same_scale = np.repeat(~bad_s, 16, axis=1)
        bad = (cg != cr) & same_scale
        assert bad.mean() < 1e-3, f"rows {r0}..{r1}: {bad.sum()} code differences"
        a, b = cg[bad], cr[bad]
        # one step of the same sign, or a zero whose sign the accumulation
        # order decides (a value within the accumulation error of 0)
        adj = (((a & 8) == (b & 8)) & (np.abs((a & 7).astype(int) - (b & 7).astype(int)) == 1)) | \
              (((a & 7) == 0) & ((b & 7) == 0))
        assert adj.all(), f"code differences larger than one step: gpu {a[~adj][:8]} oracle {b[~adj][:8]}"


def test_gemm_error_bits_clear():
    x, w = _exact_operands(256, 256, 128, 9)
    G.glu_quant_device_errors(clear=True)
    G.gemm(x, w, act=G.ACT_GELU_TANH, fmt=G.FMT_NVFP4)
    torch.cuda.synchronize()
    st, f, b = G.glu_quant_device_errors(clear=True)
    assert st == 0 and f == 0 and b == 0


def test_gemm_rejects_bad_shapes():
    x, w = _exact_operands(128, 128, 64, 10)
    with pytest.raises(G.GluQuantError):
        G.gemm(x[:, :48].contiguous(), w[:, :48].contiguous())  # K % 64
    with pytest.raises(G.GluQuantError):
        G.gemm(x, w[:192].contiguous())  # H = 96, not a multiple of 128
