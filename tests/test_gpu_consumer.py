"""The 128x4 scale layout read by a real consumer: a block-scaled GEMM.

"feat(phyai-kernel): add Thor NVFP4 GeGLU kernel for pi0.5", Supported
contract, names the scale layout only ("128x4", the layout CUTLASS and
FlashInfer read).  The oracle and the kernels write the same reading of it,
so agreement between them cannot show that the reading is the one a
block-scaled GEMM uses.  This test can: it quantises two operands with the
library (gate = the operand, up = 1, the identity gate, so h is the operand
exactly), hands the codes and the 128x4 scale buffers to torch's
block-scaled ``_scaled_mm`` (cuBLAS on the local GPU), and compares the
product with an fp64 host GEMM of the operands dequantised from the
oracle's codes and its plain row-major scales.  A wrong tile order, a wrong
order inside a tile or (NVFP4) a wrong nibble order puts scales of other
blocks under the codes, which moves the product by orders of magnitude:
the operands' 32- (16-) element blocks are scaled by independent random
powers of two.
"""
import numpy as np
import pytest
import torch

import oracle as O
from parity_util import host, host_bits

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import fp4_quant_gb300 as G  # noqa: E402

DEV = torch.device("cuda:0")


def _blocky(rows, cols, block, kmin, kmax, seed):
    """bf16 [rows, cols]: N(0,1) times 2^k, k drawn per block of `block`
    consecutive columns (exact in bf16: a power-of-two factor)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(rows, cols, generator=g)
    k = torch.randint(kmin, kmax + 1, (rows, cols // block), generator=g).to(torch.float32)
    x = x * torch.exp2(k).repeat_interleave(block, dim=1)
    return x.to(torch.bfloat16).to(DEV)


def _quantise(x, fmt):
    ones = torch.ones_like(x)
    return G.fwd(x, ones, act=G.ACT_IDENTITY, fmt=fmt, mode=G.MODE_ROW)


def _scaled_mm(a, b, sa, sb, out_dtype):
    try:
        return torch._scaled_mm(a, b.t(), scale_a=sa, scale_b=sb, out_dtype=out_dtype)
    except (RuntimeError, TypeError, NotImplementedError) as e:
        pytest.skip(f"torch._scaled_mm refused the block-scaled call: {str(e).splitlines()[0]}")


def _check(C, ref, absref, rel, what):
    C = C.double().cpu().numpy()
    err = np.abs(C - ref)
    tol = rel * np.abs(ref) + 1e-5 * absref + 1e-30
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} products off "
                           f"(worst {float((err / np.maximum(absref, 1e-30)).max()):.3g} of sum|a||b|)")


@pytest.mark.parametrize("M,N,K", [(384, 256, 640), (256, 384, 512)])
def test_mxfp8_128x4_scales_in_a_block_scaled_gemm(M, N, K):
    # 3 (2) row tiles and K/32 = 20 (16) scale columns = 5 (4) column tiles
    A = _blocky(M, K, 32, -12, 12, 1)
    B = _blocky(N, K, 32, -12, 12, 2)
    qa, qb = _quantise(A, G.FMT_MXFP8_128X4), _quantise(B, G.FMT_MXFP8_128X4)
    torch.cuda.synchronize()
    C = _scaled_mm(qa["q_row"].view(torch.float8_e4m3fn), qb["q_row"].view(torch.float8_e4m3fn),
                   qa["s_row"].view(torch.float8_e8m0fnu), qb["s_row"].view(torch.float8_e8m0fnu),
                   torch.float32)
    torch.cuda.synchronize()

    # the host side: the oracle's codes and plain row-major scales
    deq = []
    for X, q in ((A, qa), (B, qb)):
        ones = np.full(host_bits(X).shape, 0x3F80, np.uint16)
        r = O.glu_fwd(host_bits(X), ones, act=O.IDENTITY, fmt=O.MXFP8, mode=O.ROW)
        assert np.array_equal(host(q["q_row"]), r["q_row"]), "codes differ from the oracle's"
        assert np.array_equal(host(q["s_row"]), O.scales_128x4(r["s_row"])), "128x4 buffer differs"
        s = np.repeat(O.e8m0_decode(r["s_row"]).astype(np.float64), 32, axis=1)
        deq.append(O.e4m3_decode(r["q_row"]).astype(np.float64) * s)
    ref = deq[0] @ deq[1].T
    absref = np.abs(deq[0]) @ np.abs(deq[1]).T
    # fp32 output, fp32 accumulation: a few ulps of sum |a||b| at K <= 640
    _check(C, ref, absref, 1e-6, "mxfp8")


@pytest.mark.parametrize("M,N,K", [(384, 256, 512)])
def test_nvfp4_128x4_scales_and_nibbles_in_a_block_scaled_gemm(M, N, K):
    # K/16 = 32 scale columns = 8 column tiles; block amax/6 stays inside E4M3
    A = _blocky(M, K, 16, -3, 3, 3)
    B = _blocky(N, K, 16, -3, 3, 4)
    qa, qb = _quantise(A, G.FMT_NVFP4), _quantise(B, G.FMT_NVFP4)
    torch.cuda.synchronize()
    f4 = getattr(torch, "float4_e2m1fn_x2", None)
    if f4 is None:
        pytest.skip("this torch has no float4_e2m1fn_x2")
    C = _scaled_mm(qa["q_row"].view(f4), qb["q_row"].view(f4),
                   qa["s_row"].view(torch.float8_e4m3fn), qb["s_row"].view(torch.float8_e4m3fn),
                   torch.bfloat16)
    torch.cuda.synchronize()

    deq = []
    for X, q in ((A, qa), (B, qb)):
        ones = np.full(host_bits(X).shape, 0x3F80, np.uint16)
        r = O.glu_fwd(host_bits(X), ones, act=O.IDENTITY, fmt=O.NVFP4)
        assert np.array_equal(host(q["q_row"]), r["out"]), "packed codes differ from the oracle's"
        assert np.array_equal(host(q["s_row"]), r["s_nvfp4"]), "128x4 scale buffer differs"
        rows = X.shape[0]
        # element 2i in the low nibble (the oracle's packing)
        codes = np.stack([r["out"] & 0xF, r["out"] >> 4], axis=-1).reshape(rows, -1)
        # the plain [rows, K/16] scales, straight from the block amax (h is
        # the operand itself), not through any reading of the layout
        h = (host_bits(X).astype(np.uint32) << 16).view(np.float32)
        plain = O.nvfp4_scale(np.abs(h).reshape(rows, K // 16, 16).max(axis=2))
        s = np.repeat(O.e4m3_decode(plain).astype(np.float64), 16, axis=1)
        deq.append(O.e2m1_decode(codes).astype(np.float64) * s)
    ref = deq[0] @ deq[1].T
    absref = np.abs(deq[0]) @ np.abs(deq[1]).T
    # bf16 output: one rounding of the fp32 sum
    _check(C, ref, absref, 2.0 ** -8, "nvfp4")
