"""Pins of the oracle's gate/up GEMM path (no GPU).

The path ("feat(phyai-kernel): add Thor NVFP4 GeGLU kernel for pi0.5",
Summary: merged gate/up projection, GeGLU fold, quantised store) composes a
GEMM of bf16 operands with the forward quantiser.  The GEMM step is pinned
against exact integer arithmetic; the composition against the already
pinned forward oracle, fed the projection itself whenever every entry of the
projection is a bf16 value (operands chosen so that it is): any slip in the
pairing of gate and up (interleaved or split weight rows), in the activation
or in the quantiser shows up as a difference.
"""
import numpy as np
import pytest

import oracle as O


def _bf16_bits(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _val(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _small_int_operands(M, H, K, seed, density=0.25):
    """X in {-3..3}/4, W in {-3..3}/8 (bf16-exact), sparse enough that every
    entry of C = X W^T is a multiple of 1/32 below 2^3 in magnitude, so that
    C itself is a bf16 value (at most 8 significant bits)."""
    rng = np.random.default_rng(seed)
    x = rng.integers(-3, 4, (M, K)) * (rng.random((M, K)) < density)
    w = rng.integers(-3, 4, (2 * H, K)) * (rng.random((2 * H, K)) < density)
    return x, w, _bf16_bits(x / 4.0), _bf16_bits(w / 8.0)


def test_gemm_step_is_the_exact_integer_product():
    x, w, xb, wb = _small_int_operands(16, 64, 256, 1, density=1.0)
    r = O.gemm_glu_fwd(xb, wb, act=O.IDENTITY, fmt=O.NVFP4, want_c=True)
    exact = (x.astype(np.int64) @ w.astype(np.int64).T) / 32.0  # (x/4)(w/8)
    assert np.array_equal(r["c"].astype(np.float64), exact)


def test_gemm_step_rounds_the_double_sum_once():
    # general bf16 operands: C is the double sum rounded to fp32
    rng = np.random.default_rng(2)
    xb = _bf16_bits(rng.standard_normal((8, 128)))
    wb = _bf16_bits(rng.standard_normal((64, 128)))
    r = O.gemm_glu_fwd(xb, wb, act=O.IDENTITY, fmt=O.MXFP8, want_c=True)
    ref = (_val(xb).astype(np.float64) @ _val(wb).astype(np.float64).T).astype(np.float32)
    # the double sums of 128 exact products agree with numpy's to far below
    # an fp32 ulp, so the rounded values agree (up to a rare double-rounding
    # tie, none with this seed)
    assert np.array_equal(r["c"], ref)


def _c_bits_ok(c):
    """Every entry of C is exactly a bf16 value."""
    return np.array_equal(_val(_bf16_bits(c)), c)


@pytest.mark.parametrize("act", [O.SILU, O.GELU_TANH, O.RELU, O.IDENTITY, O.GELU_ERF],
                         ids=["silu", "gelu", "relu", "identity", "gelu_erf"])
@pytest.mark.parametrize("fmt", [O.NVFP4, O.MXFP8, O.MXFP8_128X4], ids=["nvfp4", "mxfp8", "mxfp8_128x4"])
@pytest.mark.parametrize("layout", [O.INTERLEAVED, O.SPLIT], ids=["inter", "split"])
def test_gemm_path_equals_forward_path_on_its_projection(act, fmt, layout):
    M, H, K = 200, 96, 64
    _, _, xb, wb = _small_int_operands(M, H, K, 3)
    r = O.gemm_glu_fwd(xb, wb, act=act, fmt=fmt, layout=layout, want_c=True, want_h=True)
    c = r["c"]
    assert _c_bits_ok(c)
    cb = _bf16_bits(c)
    if layout == O.INTERLEAVED:
        ref = O.glu_fwd(cb, act=act, fmt=fmt, layout=O.INTERLEAVED, want_h=True)
    else:
        ref = O.glu_fwd(np.ascontiguousarray(cb[:, :H]), np.ascontiguousarray(cb[:, H:]), act=act, fmt=fmt,
                        layout=O.SPLIT, want_h=True)
    assert np.array_equal(r["h"], ref["h"])
    if fmt == O.NVFP4:
        assert np.array_equal(r["q"], ref["out"]) and np.array_equal(r["s"], ref["s_nvfp4"])
    else:
        assert np.array_equal(r["q"], ref["q_row"]) and np.array_equal(r["s"], ref["s_row"])


def test_gemm_path_pairs_gate_and_up_by_layout():
    # one hand-made case: W rows (2j, 2j+1) interleaved vs (j, H+j) split
    # give the same h when the split W is the interleaved one re-ordered
    M, H, K = 4, 32, 64
    _, _, xb, wb = _small_int_operands(M, H, K, 4, density=0.5)
    ri = O.gemm_glu_fwd(xb, wb, act=O.GELU_TANH, fmt=O.MXFP8, layout=O.INTERLEAVED, want_h=True)
    ws = np.ascontiguousarray(np.concatenate([wb[0::2], wb[1::2]]))
    rs = O.gemm_glu_fwd(xb, ws, act=O.GELU_TANH, fmt=O.MXFP8, layout=O.SPLIT, want_h=True)
    assert np.array_equal(ri["h"], rs["h"]) and np.array_equal(ri["q"], rs["q"])
    # and h is act(gate) * up of the pairs, by the scalar activation
    c = (_val(xb).astype(np.float64) @ _val(wb).astype(np.float64).T)
    g, u = c[:, 0::2].astype(np.float32), c[:, 1::2].astype(np.float32)
    want = (O.act(O.GELU_TANH, g.astype(np.float64)) * u.astype(np.float64)).astype(np.float32)
    assert np.array_equal(ri["h"], want)
