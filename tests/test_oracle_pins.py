"""Pins of the CPU oracle against things other than itself.

Each test fixes a piece of the oracle to an independent source: a hand-worked
value (tests/golden/format_values.txt), a closed form, an exhaustive
comparison against independent encoder implementations (ml_dtypes, torch),
brute-force nearest-value search, a high-precision (mpmath) evaluation of the
activation in the pages' tanh form, or an invariant of the method.  A plausible
mistake in the oracle (a dropped term, a wrong sign, a swapped operand, a
transposed layout, a wrong tie rule) fails at least one of them.
"""
import math
import os

import ml_dtypes
import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "format_values.txt")


def _parse_float(s):
    return float.fromhex(s) if "0x" in s and "p" in s else float(s)


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if line:
            kind, v, exp = line.split()
            rows.append((kind, _parse_float(v), int(exp, 16)))
    return rows


@pytest.mark.parametrize("kind,value,expected", _golden_rows())
def test_hand_worked_values(kind, value, expected):
    fn = {"e8m0": O.e8m0_rceil, "e4m3": O.e4m3_encode,
          "nvfp4s": O.nvfp4_scale, "e2m1": O.e2m1_encode}[kind]
    assert int(fn([value])[0]) == expected


# ---------------------------------------------------------------- encoders --

def _sweep_against(kind, first, n, ref_dtype, chunk=1 << 25):
    """Compare oracle codes for all fp32 bit patterns first..first+n-1
    against a cast through ref_dtype."""
    done = 0
    while done < n:
        m = min(chunk, n - done)
        start = first + done
        ours = O.encode_bits(kind, start, m)
        vals = np.arange(start, start + m, dtype=np.uint64).astype(np.uint32).view(np.float32)
        ref = vals.astype(ref_dtype).view(np.uint8)
        if kind == 1:
            ref = ref & 0xF
        bad = np.nonzero(ours != ref)[0]
        assert bad.size == 0, (hex(int(vals.view(np.uint32)[bad[0]])), ours[bad[0]], ref[bad[0]])
        done += m


@pytest.mark.slow
def test_e4m3_exhaustive_nonnegative_vs_ml_dtypes():
    # every non-negative fp32 up to and including 448
    _sweep_against(0, 0, 0x43E00000 + 1, ml_dtypes.float8_e4m3fn)


@pytest.mark.slow
def test_e2m1_exhaustive_nonnegative_vs_ml_dtypes():
    # every non-negative fp32 up to and including 6
    _sweep_against(1, 0, 0x40C00000 + 1, ml_dtypes.float4_e2m1fn)


def test_negative_values_mirror_positive():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 0x43E00001, 2_000_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    assert np.array_equal(O.e4m3_encode(-v), O.e4m3_encode(v) | 0x80)
    b2 = rng.integers(0, 0x40C00001, 2_000_000, dtype=np.uint64).astype(np.uint32)
    v2 = b2.view(np.float32)
    assert np.array_equal(O.e2m1_encode(-v2), O.e2m1_encode(v2) | 0x8)
    # and against ml_dtypes on the negative side too
    ref = (-v).astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(O.e4m3_encode(-v), ref)


def test_e4m3_vs_torch_float8():
    g = torch.Generator().manual_seed(7)
    x = (torch.rand(4_000_000, generator=g) * 2 - 1) * 448
    x = torch.cat([x, x * 1e-3, x * 1e-5, torch.tensor([0.0, -0.0, 448.0, -448.0])])
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x.numpy()), ref)


def _e4m3_values_from_spec():
    """All finite non-negative E4M3 magnitudes with their codes, built from
    the format description (not from the oracle)."""
    out = []
    for ex in range(16):
        for m in range(8):
            if ex == 15 and m == 7:
                continue
            val = m * 2.0 ** -9 if ex == 0 else (1 + m / 8) * 2.0 ** (ex - 7)
            out.append((val, (ex << 3) | m))
    return out


def _nearest_even(values_codes, a):
    best = None
    for val, code in values_codes:
        d = abs(val - a)
        if best is None or d < best[0] or (d == best[0] and (code & 1) == 0):
            best = (d, code)
    return best[1]


def test_e4m3_brute_force_nearest():
    vc = _e4m3_values_from_spec()
    rng = np.random.default_rng(3)
    # random magnitudes over the whole range, plus every exact midpoint
    sample = list(np.exp2(rng.uniform(-12, 8.8, 3000)).astype(np.float32))
    vals = sorted(v for v, _ in vc)
    sample += [np.float32((a + b) / 2) for a, b in zip(vals, vals[1:])]
    sample = [s for s in sample if s <= 448]
    ours = O.e4m3_encode(np.array(sample, np.float32))
    for s, c in zip(sample, ours):
        assert c == _nearest_even(vc, float(s)), (s, c)


def test_e2m1_brute_force_nearest_and_roundtrip():
    vc = [(0.0, 0), (0.5, 1), (1.0, 2), (1.5, 3), (2.0, 4), (3.0, 5), (4.0, 6), (6.0, 7)]
    grid = np.linspace(0, 6, 6001).astype(np.float32)
    mids = np.array([(a[0] + b[0]) / 2 for a, b in zip(vc, vc[1:])], np.float32)
    sample = np.concatenate([grid, mids])
    ours = O.e2m1_encode(sample)
    for s, c in zip(sample, ours):
        assert c == _nearest_even(vc, float(s))
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(O.e2m1_encode(O.e2m1_decode(codes)), codes)


def test_e4m3_decode_encode_roundtrip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(O.e4m3_encode(O.e4m3_decode(codes)), codes)
    ref = codes.view(ml_dtypes.float8_e4m3fn).astype(np.float32)
    assert np.array_equal(O.e4m3_decode(codes), ref)


def test_e8m0_closed_form():
    rng = np.random.default_rng(5)
    ex = rng.integers(-149, 128, 200_000)
    mant = rng.uniform(1, 2, 200_000)
    amax = (mant * np.exp2(ex.astype(np.float64))).astype(np.float32)
    amax = amax[np.isfinite(amax) & (amax > 0)]
    edges = np.array([448.0 * 2.0 ** k for k in range(-140, 121)], np.float64)
    edges = edges[(edges < 3.4e38) & (edges > 1e-45)].astype(np.float32)
    amax = np.concatenate([amax, edges, np.nextafter(edges, np.float32(np.inf)),
                           np.nextafter(edges, np.float32(0))])
    s = O.e8m0_rceil(amax).astype(np.int64)
    for a, b in zip(amax.astype(np.float64), s):
        e = int(b) - 127
        assert a <= 448.0 * 2.0 ** e, (a, e)
        if e > -127:
            assert a > 448.0 * 2.0 ** (e - 1), (a, e)
    # the same bytes from the fp32 bit fields: biased exponent - 8, plus one
    # when the significand exceeds 1.75 (448 = 1.75 * 2^8); floor at 0
    nz = amax[amax >= np.float32(2.0 ** -126)]
    u = nz.view(np.uint32).astype(np.int64)
    byte = np.maximum((u >> 23) - 8 + ((u & 0x7FFFFF) > 0x600000), 0)
    assert np.array_equal(O.e8m0_rceil(nz).astype(np.int64), byte)
    assert O.e8m0_rceil([0.0])[0] == 0
    assert O.e8m0_rceil([np.inf])[0] == 0xFF and O.e8m0_rceil([np.nan])[0] == 0xFF


def test_nvfp4_scale_is_nearest_e4m3_of_quotient():
    vc = _e4m3_values_from_spec()
    rng = np.random.default_rng(9)
    amax = np.exp2(rng.uniform(-14, 12, 2000)).astype(np.float32)
    ours = O.nvfp4_scale(amax)
    for a, c in zip(amax, ours):
        q = float(np.float32(a) / np.float32(6.0))
        exp = 0x7E if q >= 448 else _nearest_even(vc, q)
        assert c == exp, (a, c, exp)


def test_bf16_rne():
    rng = np.random.default_rng(11)
    x = rng.standard_normal(1_000_000).astype(np.float32) * np.exp2(rng.integers(-60, 60, 1_000_000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_rne(x), ref)


# -------------------------------------------------------------- activation --

def _all_bf16_in(lo, hi):
    b = np.arange(0, 1 << 16, dtype=np.uint32)
    v = (b << 16).view(np.float32)
    v = v[np.isfinite(v) & (v >= lo) & (v <= hi)]
    return np.unique(v.astype(np.float64))


def test_activation_special_values():
    for kind in (O.SILU, O.GELU_TANH):
        assert O.act(kind, [0.0])[0] == 0.0
        assert O.act_grad(kind, [0.0])[0] == 0.5
        assert np.float32(O.act(kind, [60.0])[0]) == np.float32(60.0)
        assert np.float32(O.act_grad(kind, [60.0])[0]) == np.float32(1.0)
        # sign of tiny outputs in the negative tail
        assert math.copysign(1, O.act(kind, [-500.0])[0]) == -1


def test_activation_vs_mpmath_tanh_form():
    mpmath = pytest.importorskip("mpmath")
    # 1 + tanh(y) cancels down to e^(2y); at x = -14 that is e^-437, so the
    # reference needs a few hundred digits to keep its own relative precision
    mpmath.mp.dps = 420
    c = mpmath.sqrt(2 / mpmath.pi)
    a = mpmath.mpf("0.044715")

    def gelu(x):
        return x / 2 * (1 + mpmath.tanh(c * (x + a * x ** 3)))

    def silu(x):
        return x / (1 + mpmath.exp(-x))

    for kind, f, lo, hi in ((O.SILU, silu, -120.0, 120.0), (O.GELU_TANH, gelu, -14.0, 14.0)):
        xs = _all_bf16_in(lo, hi)[::7]
        ours, ours_d = O.act(kind, xs), O.act_grad(kind, xs)
        for x, y, dy in zip(xs, ours, ours_d):
            X = mpmath.mpf(float(x))
            ref = f(X)
            dref = mpmath.diff(f, X)
            # exp(t) has condition number |t|: the double evaluation's relative
            # error grows with the argument (|t| ~ 0.07 |x|^3 for GELU); any
            # formula mistake is O(1), far above this bound
            cond = 1.0 + abs(float(x)) + (0.1 * abs(float(x)) ** 3 if kind == O.GELU_TANH else 0.0)
            assert abs(y - float(ref)) <= 1e-15 * cond * abs(float(ref)) + 1e-300, (kind, x)
            # act' has zeros; bound the error by its term magnitudes
            scale = abs(float(dref)) + 1e-13 * (1 + abs(float(x)))
            assert abs(dy - float(dref)) <= 1e-13 * cond * scale, (kind, x, dy, float(dref))


def test_activation_vs_torch_float64():
    # torch evaluates the tanh form, whose 1 + tanh(y) cancels for x << 0;
    # stay where that library form is itself accurate (the tail is pinned
    # against mpmath above)
    x = torch.linspace(-3, 20, 20001, dtype=torch.float64)
    assert np.allclose(O.act(O.SILU, x.numpy()), torch.nn.functional.silu(x).numpy(), rtol=1e-14, atol=0)
    ref = torch.nn.functional.gelu(x, approximate="tanh").numpy()
    assert np.allclose(O.act(O.GELU_TANH, x.numpy()), ref, rtol=1e-12, atol=1e-300)
    # derivatives through autograd of the library forms
    for kind, fn in ((O.SILU, torch.nn.functional.silu),
                     (O.GELU_TANH, lambda t: torch.nn.functional.gelu(t, approximate="tanh"))):
        t = x.clone().requires_grad_(True)
        fn(t).sum().backward()
        assert np.allclose(O.act_grad(kind, x.numpy()), t.grad.numpy(), rtol=1e-11, atol=1e-14)


def test_activation_gradient_finite_differences():
    xs = np.linspace(-9, 9, 1801)
    h = 1e-5
    for kind in (O.SILU, O.GELU_TANH):
        fd = (O.act(kind, xs + h) - O.act(kind, xs - h)) / (2 * h)
        assert np.allclose(O.act_grad(kind, xs), fd, rtol=0, atol=1e-8)


# ---------------------------------------------------------- the full path --

def _bf16_bits(x):
    return np.asarray(x, np.float32).astype(ml_dtypes.bfloat16).view(np.uint16)


def test_exact_activation_blocks_mxfp8_row():
    # gate = 32: sigmoid(32) rounds to 1 in fp32 and h = 32 * up exactly, so
    # every block below has a hand-computable scale and codes.
    N = 32 * 6
    up = np.zeros((2, N), np.float32)
    up[0, 0] = 14.0                 # block 0: amax 448 -> scale 127, code 0x7E
    up[0, 32] = 28.0                # block 1: amax 896 -> 128, 896/2 = 448 -> 0x7E
    up[0, 64] = 2.0 ** -5           # block 2: amax 1 -> 119, v = 256 -> 0x78
    up[0, 96] = 14.0                # block 3: e = 0 ...
    up[0, 97] = 2.0 ** -14          # ... h = 2^-9 -> subnormal code 0x01
    up[0, 98] = 3 * 2.0 ** -15      # ... h = 3*2^-10 -> tie -> 0x02
    up[0, 99] = 17 * 2.0 ** -9      # ... h = 1.0625 -> tie -> 0x38
    up[0, 100] = -(2.0 ** -16)      # ... h = -2^-11 -> 0x80
    up[0, 128:160] = 0.0            # block 4: all zero -> scale 0, codes 0
    up[0, 160:192] = -0.0           # block 5: all -0 -> scale 0, codes 0x80
    up[0, 160] = 0.0
    up[1] = up[0] * -1
    gate = np.full((2, N), 32.0, np.float32)
    for kind in (O.SILU, O.GELU_TANH):
        r = O.glu_fwd(_bf16_bits(gate), _bf16_bits(up), act=kind, fmt=O.MXFP8, mode=O.ROW, want_h=True)
        assert np.array_equal(r["h"][0], (32 * up[0]).astype(np.float32))
        q, s = r["q_row"], r["s_row"]
        assert list(s[0]) == [127, 128, 119, 127, 0, 0]
        assert q[0, 0] == 0x7E and q[0, 32] == 0x7E and q[0, 64] == 0x78
        assert list(q[0, 96:101]) == [0x7E, 0x01, 0x02, 0x38, 0x80]
        assert np.all(q[0, 101:128] == 0) and np.all(q[0, 1:32] == 0)
        assert np.all(q[0, 128:160] == 0)
        assert q[0, 160] == 0 and np.all(q[0, 161:192] == 0x80)
        # negated up: same scales, sign bits flipped (zeros flip too)
        assert np.array_equal(s[1], s[0])
        assert np.array_equal(q[1], q[0] ^ 0x80)


def test_sign_of_zero_product():
    gate = _bf16_bits(np.full((1, 32), -1.0))
    up = _bf16_bits(np.zeros((1, 32)))
    r = O.glu_fwd(gate, up, act=O.SILU, fmt=O.MXFP8, mode=O.ROW)
    assert np.all(r["q_row"] == 0x80)  # silu(-1) < 0, times +0 = -0


def test_exact_activation_nvfp4_interleaved():
    H = 64
    x = np.zeros((1, 2 * H), np.float32)
    x[0, 0::2] = 32.0               # gate columns
    ups = np.zeros(H, np.float32)
    ups[0:4] = [6 / 32, -0.5 / 32, 0.25 / 32, 0.75 / 32]   # block 0: amax 6 -> s 1.0
    ups[16] = 12 / 32                                      # block 1: amax 12 -> s 2.0
    ups[17] = 3 / 32                                       # h = 3 -> v = 1.5 -> 0x3
    ups[32] = 2.0 ** -20                                   # block 2: s -> 0, codes 0
    ups[33] = -(2.0 ** -20)                                # -> sign-kept zero 0x8
    ups[48:64] = 0.0                                       # block 3: zeros
    x[0, 1::2] = ups
    r = O.glu_fwd(_bf16_bits(x), act=O.GELU_TANH, fmt=O.NVFP4, layout=O.INTERLEAVED)
    q, s = r["out"], r["s_nvfp4"]
    # element 2i in the low nibble, 2i+1 in the high nibble
    assert q[0, 0] == (0x7 | (0x9 << 4))      # 6 -> 7, -0.5 -> 0x9
    assert q[0, 1] == (0x0 | (0x2 << 4))      # 0.25 tie -> 0, 0.75 tie -> 1.0
    assert q[0, 8] == (0x7 | (0x3 << 4))      # 12/2 = 6 -> 7, 3/2 = 1.5 -> 3
    assert q[0, 16] == (0x0 | (0x8 << 4))
    # scales at the 128x4 offsets of row 0, columns 0..3
    assert [s[O.swizzle_offset(0, c, 4)] for c in range(4)] == [0x38, 0x40, 0x00, 0x00]
    # padding rows 1..127 are zero
    assert s.sum() == 0x38 + 0x40


def test_swizzle_is_bijection_on_padded_domain():
    for M, N in ((128, 64), (784, 16384 // 64 * 64), (200, 80), (1, 16)):
        C = N // 16
        rp, cp = -(-M // 128) * 128, -(-C // 4) * 4
        offs = np.array([O.swizzle_offset(r, c, cp) for r in range(rp) for c in range(cp)]) \
            if rp * cp < 300_000 else None
        if offs is None:
            continue
        assert np.array_equal(np.sort(offs), np.arange(rp * cp))
    assert O.swizzle_offset(0, 0, 8) == 0
    assert O.swizzle_offset(1, 0, 8) == 16
    assert O.swizzle_offset(32, 0, 8) == 4
    assert O.swizzle_offset(0, 1, 8) == 1
    assert O.swizzle_offset(0, 4, 8) == 512
    assert O.swizzle_offset(128, 0, 8) == 1024


def _rand_inputs(M, N, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    g = _bf16_bits(rng.standard_normal((M, N)) * scale)
    u = _bf16_bits(rng.standard_normal((M, N)) * scale)
    return g, u


@pytest.mark.parametrize("kind", [O.SILU, O.GELU_TANH])
def test_both_equals_row_and_col(kind):
    g, u = _rand_inputs(96, 160, 1)
    b = O.glu_fwd(g, u, act=kind, fmt=O.MXFP8, mode=O.BOTH)
    r = O.glu_fwd(g, u, act=kind, fmt=O.MXFP8, mode=O.ROW)
    c = O.glu_fwd(g, u, act=kind, fmt=O.MXFP8, mode=O.COL)
    for k in ("q_row", "s_row"):
        assert np.array_equal(b[k], r[k])
    for k in ("q_col", "s_col"):
        assert np.array_equal(b[k], c[k])


@pytest.mark.parametrize("kind", [O.SILU, O.GELU_TANH])
def test_col_is_row_of_transpose(kind):
    g, u = _rand_inputs(64, 96, 2)
    c = O.glu_fwd(g, u, act=kind, fmt=O.MXFP8, mode=O.COL)
    rt = O.glu_fwd(np.ascontiguousarray(g.T), np.ascontiguousarray(u.T), act=kind,
                   fmt=O.MXFP8, mode=O.ROW)
    # colwise codes are stored [N, M]: exactly the rowwise codes of the transpose
    assert np.array_equal(c["q_col"], rt["q_row"])
    assert np.array_equal(c["s_col"], rt["s_row"])


def test_layout_invariance():
    g, u = _rand_inputs(64, 128, 3)
    M, N = g.shape
    packed = np.concatenate([g, u], axis=1)               # [gate | up], ld = 2N
    inter = np.empty((M, 2 * N), np.uint16)
    inter[:, 0::2], inter[:, 1::2] = g, u
    for fmt, mode in ((O.MXFP8, O.BOTH), (O.NVFP4, O.ROW), (O.FP32, O.ROW)):
        a = O.glu_fwd(g, u, act=O.GELU_TANH, fmt=fmt, mode=mode)
        b = O.glu_fwd(packed[:, :N], packed[:, N:], act=O.GELU_TANH, fmt=fmt, mode=mode)
        c = O.glu_fwd(inter, act=O.GELU_TANH, fmt=fmt, mode=mode, layout=O.INTERLEAVED)
        for k in a:
            if a[k] is not None:
                assert np.array_equal(a[k], b[k]) and np.array_equal(a[k], c[k]), (fmt, k)


def test_row_chunk_invariance_and_determinism():
    g, u = _rand_inputs(256, 64, 4)
    full = O.glu_fwd(g, u, act=O.SILU, fmt=O.MXFP8, mode=O.BOTH, nthreads=3)
    again = O.glu_fwd(g, u, act=O.SILU, fmt=O.MXFP8, mode=O.BOTH, nthreads=1)
    top = O.glu_fwd(g[:128], u[:128], act=O.SILU, fmt=O.MXFP8, mode=O.BOTH)
    bot = O.glu_fwd(g[128:], u[128:], act=O.SILU, fmt=O.MXFP8, mode=O.BOTH)
    for k in full:
        assert np.array_equal(full[k], again[k])
    assert np.array_equal(full["q_row"], np.concatenate([top["q_row"], bot["q_row"]]))
    assert np.array_equal(full["q_col"], np.concatenate([top["q_col"], bot["q_col"]], axis=1))
    assert np.array_equal(full["s_col"], np.concatenate([top["s_col"], bot["s_col"]], axis=1))


def test_dequantisation_error_bound():
    g, u = _rand_inputs(64, 256, 5)
    r = O.glu_fwd(g, u, act=O.SILU, fmt=O.MXFP8, mode=O.ROW, want_h=True)
    h = r["h"].astype(np.float64)
    scale = np.repeat(O.e8m0_decode(r["s_row"]).astype(np.float64), 32, axis=1)
    deq = O.e4m3_decode(r["q_row"]).astype(np.float64) * scale
    v = np.abs(h / scale)
    normal = v >= 2.0 ** -6
    assert np.all(np.abs(deq - h)[normal] <= 2.0 ** -4 * np.abs(h)[normal])
    assert np.all(np.abs(deq - h)[~normal] <= 2.0 ** -10 * scale[~normal])


def test_backward_exact_activation():
    # gate = 32: act'(32) rounds to 1 and act(32) = 32 in fp32, so
    # dGate = dY*up and dUp = 32*dY exactly; they land in [dGate | dUp].
    rng = np.random.default_rng(6)
    M, N = 32, 64
    gate = np.full((M, N), 32.0, np.float32)
    up = rng.standard_normal((M, N)).astype(ml_dtypes.bfloat16).astype(np.float32)
    dy = rng.standard_normal((M, N)).astype(ml_dtypes.bfloat16).astype(np.float32)
    for kind in (O.SILU, O.GELU_TANH):
        r = O.glu_bwd(_bf16_bits(gate), _bf16_bits(up), _bf16_bits(dy), act=kind, fmt=O.FP32)
        out = r["out"]
        assert np.array_equal(out[:, :N], (dy * up).astype(np.float32))
        assert np.array_equal(out[:, N:], (32 * dy).astype(np.float32))


def test_backward_formula_against_autograd():
    g, u = _rand_inputs(32, 64, 8)
    d, _ = _rand_inputs(32, 64, 9)
    gf = torch.from_numpy(g.astype(np.uint32) << 16).view(torch.float32).double()
    uf = torch.from_numpy(u.astype(np.uint32) << 16).view(torch.float32).double()
    df = torch.from_numpy(d.astype(np.uint32) << 16).view(torch.float32).double()
    for kind, fn in ((O.SILU, torch.nn.functional.silu),
                     (O.GELU_TANH, lambda t: torch.nn.functional.gelu(t, approximate="tanh"))):
        gg = gf.clone().requires_grad_(True)
        uu = uf.clone().requires_grad_(True)
        (fn(gg) * uu * df).sum().backward()
        r = O.glu_bwd(g, u, d, act=kind, fmt=O.FP32)
        ref = torch.cat([gg.grad, uu.grad], dim=1).float().numpy()
        assert np.allclose(r["out"], ref, rtol=2e-7, atol=1e-30)


def test_fp32_mode_is_rounded_exact_value():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    g, u = _rand_inputs(4, 64, 10)
    r = O.glu_fwd(g, u, act=O.SILU, fmt=O.FP32)
    gv = (g.astype(np.uint32) << 16).view(np.float32)
    uv = (u.astype(np.uint32) << 16).view(np.float32)
    for x, y, o in zip(gv.ravel(), uv.ravel(), r["out"].ravel()):
        X = mpmath.mpf(float(x))
        exact = X / (1 + mpmath.exp(-X)) * mpmath.mpf(float(y))
        assert o == np.float32(float(exact))
    # GELU (erf) through the whole forward path, fp32 and bf16-step values
    r = O.glu_fwd(g, u, act=O.GELU_ERF, fmt=O.FP32)
    rb = O.glu_fwd(g, u, act=O.GELU_ERF | O.BF16_STEPS, fmt=O.FP32)
    for x, y, o, ob in zip(gv.ravel(), uv.ravel(), r["out"].ravel(), rb["out"].ravel()):
        X = mpmath.mpf(float(x))
        a = X * mpmath.ncdf(X)
        assert o == np.float32(float(a * mpmath.mpf(float(y))))
        assert ob == O.round_bf16(O.round_bf16(float(a)) * float(y))


def _around(m):
    """m and the floats one ulp below and above it."""
    m = np.float32(m)
    return np.array([m, np.nextafter(m, np.float32(0)), np.nextafter(m, np.float32(np.inf))], np.float32)


def test_boundary_distance():
    # 1.0625 is the midpoint between E4M3 1.0 and 1.125: distance 0; one
    # float above is 1 ulp away.
    v = np.array([1.0625, np.nextafter(np.float32(1.0625), np.float32(2)), 1.0], np.float32)
    assert list(O.boundary_ulps(O.MXFP8, v)) == [0, 1, 1 << 19]
    assert O.boundary_ulps(O.NVFP4, np.array([0.25], np.float32))[0] == 0
    assert O.boundary_ulps(O.BF16, np.array([1.0 + 2.0 ** -8], np.float32))[0] == 0


@pytest.mark.parametrize("fmt,mid", [
    (O.MXFP8, 2.0 ** -10),        # E4M3: 0 | smallest subnormal 2^-9
    (O.MXFP8, 3 * 2.0 ** -10),    # subnormals 2^-9 | 2^-8
    (O.MXFP8, 7.5 * 2.0 ** -9),   # largest subnormal 7 * 2^-9 | smallest normal 2^-6
    (O.MXFP8, 1.9375),            # binade edge 1.875 | 2
    (O.MXFP8, 432.0),             # 416 | 448 (the largest finite)
    (O.MXFP8, -3 * 2.0 ** -10),   # sign does not matter
    (O.NVFP4, 5.0),               # E2M1 4 | 6
    (O.NVFP4, 0.75),              # 0.5 | 1
], ids=["e4m3_zero_sub", "e4m3_sub", "e4m3_sub_normal", "e4m3_binade", "e4m3_top", "e4m3_neg", "e2m1_4_6",
        "e2m1_half_one"])
def test_boundary_distance_at_midpoints(fmt, mid):
    """Each rounding midpoint is at distance 0 and its two fp32 neighbours
    at distance 1 (also where the midpoint is a power of two, so that the
    neighbour below is half an ulp of the one above away)."""
    assert list(O.boundary_ulps(fmt, _around(mid))) == [0, 1, 1]


def test_boundary_distance_far_from_midpoints():
    # worked by hand, counting fp32 values between the value and its nearest
    # midpoint: E4M3 2^-9 (code 1) is 2^-10 below the midpoint 3 * 2^-10,
    # 2^22 floats of spacing 2^-32 (and 2^23 above the midpoint 2^-10: the
    # whole binade [2^-10, 2^-9))
    v = np.array([2.0 ** -9, 6.0, 100.0], np.float32)
    assert list(O.boundary_ulps(O.MXFP8, v[:1])) == [1 << 22]
    # E2M1 6: nearest midpoint 5, (6 - 5) / 2^-21 (the spacing in [4, 8));
    # 100 (saturates to 6; no midpoint above 5): [5, 8) at 2^-21, then the
    # whole binades [8, 16), [16, 32), [32, 64) at 2^23 floats each, then
    # [64, 100) at 2^-17
    spans = 3 * 2 ** 21 + 3 * 2 ** 23 + 36 * 2 ** 17
    assert list(O.boundary_ulps(O.NVFP4, v[1:])) == [1 << 21, spans]


def test_oracle_rejects_unsupported_arguments():
    g, u = _rand_inputs(40, 48, 11)
    with pytest.raises(ValueError):
        O.glu_fwd(g, u, act=O.SILU, fmt=O.MXFP8, mode=O.ROW)     # N % 32
    g, u = _rand_inputs(40, 64, 11)
    with pytest.raises(ValueError):
        O.glu_fwd(g, u, act=O.SILU, fmt=O.MXFP8, mode=O.COL)     # M % 32
    with pytest.raises(ValueError):
        O.glu_fwd(g, u, act=O.SILU, fmt=O.NVFP4, mode=O.BOTH)


def test_scales_128x4_layout():
    """The MXFP8 128x4 scale output: S [R, C] re-laid with zero padding.
    Offsets worked by hand from the layout's definition (128 x 4 tiles,
    row-tile-major, 512 bytes; (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4
    inside a tile)."""
    R, C = 160, 25                      # padded to 256 x 28: 2 x 7 tiles
    rng = np.random.default_rng(5)
    S = rng.integers(1, 256, size=(R, C), dtype=np.uint8)
    out = O.scales_128x4(S)
    assert out.shape == (256 * 28,)
    hand = {(0, 0): 0, (1, 0): 16, (31, 0): 496, (32, 0): 4, (96, 0): 12, (0, 1): 1,
            (0, 3): 3, (0, 4): 512, (0, 24): 6 * 512, (127, 3): 31 * 16 + 12 + 3,
            (128, 0): 7 * 512, (159, 24): (7 + 6) * 512 + 31 * 16 + 0 * 4 + 0}
    for (r, c), off in hand.items():
        assert out[off] == S[r, c], (r, c)
    # every real scale lands once, every other byte is padding (zero)
    r = np.arange(R)[:, None]
    c = np.arange(C)[None, :]
    off = ((r // 128) * 7 + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)
    assert len(np.unique(off)) == R * C
    assert np.array_equal(out[off], S)
    mask = np.ones(out.shape, bool)
    mask[off.ravel()] = False
    assert not out[mask].any()


def test_mxfp8_128x4_is_mxfp8_with_relaid_scales():
    """The oracle's 128x4 format: codes equal plain MXFP8's, scales equal
    the plain scale matrices re-laid (rowwise [M, W/32], colwise [W, M/32])."""
    rng = np.random.default_rng(9)
    M, N = 96, 160
    g = (rng.standard_normal((M, N)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    u = (rng.standard_normal((M, N)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    a = O.glu_fwd(g, u, act=O.SILU, fmt=O.MXFP8, mode=O.BOTH)
    b = O.glu_fwd(g, u, act=O.SILU, fmt=O.MXFP8_128X4, mode=O.BOTH)
    assert np.array_equal(a["q_row"], b["q_row"]) and np.array_equal(a["q_col"], b["q_col"])
    assert b["s_row"].shape == (128 * 8,) and b["s_col"].shape == (256 * 4,)
    assert np.array_equal(b["s_row"], O.scales_128x4(a["s_row"]))
    assert np.array_equal(b["s_col"], O.scales_128x4(a["s_col"]))


def test_nvfp4_global_scale_hand_worked():
    """Global encode scale G = 2688 / amax, values scaled once, then the
    unit-global-scale rule.  gate = 32 makes h = 32 * up exactly; with the
    tensor amax 96 (up = 3), G = 28: v = 2688 and 896 -> block scale
    E4M3(2688 / 6) = 448 (0x7E), codes 6 (0x7) and 2 (0x4)."""
    assert O.nvfp4_global_scale(96.0) == np.float32(28.0)
    assert O.nvfp4_global_scale(0.0) == 1.0 and O.nvfp4_global_scale(float("inf")) == 1.0
    M, N = 1, 16
    g = np.full((M, N), 0x4200, np.uint16)            # bf16 32.0
    u = np.zeros((M, N), np.uint16)
    u[0, 0] = 0x4040                                  # 3.0 -> h = 96
    u[0, 1] = 0x3F80                                  # 1.0 -> h = 32
    r = O.glu_fwd_nvfp4_gs(g, u, act=O.SILU, amax=96.0)
    assert r["v"][0, 0] == 2688.0 and r["v"][0, 1] == 896.0
    assert r["s_nvfp4"][0] == 0x7E
    assert r["out"][0, 0] == 0x7 | (0x4 << 4)          # element 0 low nibble, 1 high
    assert not r["out"][0, 1:].any()


def test_nvfp4_power_of_two_global_scale():
    """G = 2 (tensor amax 1344) scales every value exactly: blocks whose unit
    scale is a normal E4M3 below 224 get the scale one binade up (byte + 8)
    and the same codes (v / (2 s) = h / s); G = 1 (amax 2688) is the
    unit-global-scale output itself."""
    rng = np.random.default_rng(3)
    M, N = 256, 128
    g = (rng.standard_normal((M, N)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    u = (rng.standard_normal((M, N)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    plain = O.glu_fwd(g, u, act=O.GELU_TANH, fmt=O.NVFP4)
    one = O.glu_fwd_nvfp4_gs(g, u, act=O.GELU_TANH, amax=2688.0)
    assert np.array_equal(plain["out"], one["out"]) and np.array_equal(plain["s_nvfp4"], one["s_nvfp4"])
    two = O.glu_fwd_nvfp4_gs(g, u, act=O.GELU_TANH, amax=1344.0)
    sp, s2 = plain["s_nvfp4"].astype(int), two["s_nvfp4"].astype(int)
    normal = (sp >= 0x08) & (sp < 0x76)
    assert normal.sum() > 1000
    assert np.array_equal(s2[normal], sp[normal] + 8)
    # codes of those blocks: block (r, c) holds elements 16c .. 16c + 15 of row r
    C = N // 16
    cp = -(-C // 4) * 4
    r = np.arange(M)[:, None]
    c = np.arange(C)[None, :]
    off = ((r // 128) * (cp // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)
    ok = normal[off]                                   # [M, C] blocks with a normal unit scale
    qb = lambda q: q.reshape(M, C, 8)
    assert np.array_equal(qb(two["out"])[ok], qb(plain["out"])[ok])


def _bf16_grid():
    """Every finite non-negative bf16 value, ascending, as float64."""
    pats = np.arange(0x0000, 0x7F81, dtype=np.uint32)  # +0 .. +inf
    return (pats << 16).view(np.float32).astype(np.float64)


def _nearest_bf16_brute(x: float) -> float:
    """Nearest bf16 by search over the grid, ties to the even pattern."""
    grid = _bf16_grid()
    a = abs(x)
    i = int(np.searchsorted(grid, a))
    if i < len(grid) and grid[i] == a:
        r = a
    else:
        lo, hi = grid[i - 1], grid[i]
        if hi == np.inf:  # beyond the largest finite bf16: the half-way point is 2^128 - 2^119
            r = np.inf if a >= lo + 2.0 ** 119 else lo
        else:
            dl, dh = a - lo, hi - a
            r = lo if dl < dh else hi if dh < dl else (lo if (i - 1) % 2 == 0 else hi)
    return float(np.copysign(r, x))


def test_round_bf16_against_brute_force():
    rng = np.random.default_rng(17)
    grid = _bf16_grid()
    xs = list(rng.standard_normal(300) * 10.0 ** rng.integers(-45, 38, 300))
    mids = (grid[1:-1] + grid[2:]) / 2                 # every midpoint is a tie
    xs += list(mids[rng.integers(0, len(mids) - 1, 300)])
    xs += list(np.nextafter(mids[:50], 0)) + list(np.nextafter(mids[:50], 1))
    xs += [1e-41, 9.2e-41 / 2, 2.0 ** -134, 3.3895e38, 3.396e38, 3.3966e38, 3.4e38, -2.859375, 0.0]
    for x in xs:
        assert O.round_bf16(x) == _nearest_bf16_brute(x) or (np.isnan(x)), x


def test_bf16_steps_values():
    """act | 16: h = RN_bf16(RN_bf16(act(g)) * up).  Hand-worked: silu(3) =
    2.8577224 -> bf16 2.859375 (step 1/64 in [2, 4)); times up = 3 gives
    8.578125 -> bf16 8.5625 (step 1/16 in [8, 16)), where the fp32 value is
    8.5731672."""
    g = np.array([[0x4040]], np.uint16)  # 3.0
    u = np.array([[0x4040]], np.uint16)
    h = O.glu_fwd(g, u, act=O.SILU | O.BF16_STEPS, fmt=O.FP32)["out"][0, 0]
    assert h == np.float32(8.5625)
    h32 = O.glu_fwd(g, u, act=O.SILU, fmt=O.FP32)["out"][0, 0]
    assert abs(h32 - 8.5731672) < 1e-6
    # every value is a bf16 value, and equals the two roundings done on the
    # host from the oracle's double activation
    rng = np.random.default_rng(4)
    M, N = 8, 64
    g = (rng.standard_normal((M, N)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    u = (rng.standard_normal((M, N)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    for act in (O.SILU, O.GELU_TANH):
        h = O.glu_fwd(g, u, act=act | O.BF16_STEPS, fmt=O.FP32)["out"]
        gf = (g.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        uf = (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        a = np.array([O.round_bf16(x) for x in O.act(act, gf.ravel())]).reshape(M, N)
        ref = np.array([O.round_bf16(x) for x in (a * uf).ravel()]).reshape(M, N)
        assert np.array_equal(h.astype(np.float64), ref)
        assert np.all((h.view(np.uint32) & 0xFFFF) == 0)
    # the backward has no bf16-step form
    with pytest.raises(ValueError):
        O.glu_bwd(g, u, g, act=O.SILU | O.BF16_STEPS, fmt=O.FP32)


def test_bf16_steps_agree_with_torch_eager():
    """torch's CPU bf16 silu rounds its own fp32 evaluation: it can differ
    from the correctly rounded bf16 of silu(g) only where silu(g) lies
    within a few fp32 ulps of a bf16 midpoint, i.e. almost nowhere."""
    torch = pytest.importorskip("torch")
    pats = np.arange(0, 0x10000, dtype=np.uint32)
    gf = (pats << 16).view(np.float32)
    ok = np.isfinite(gf) & (np.abs(gf) < 60)
    gb = torch.from_numpy(gf[ok].copy()).to(torch.bfloat16)
    eager = torch.nn.functional.silu(gb).float().numpy().astype(np.float64)
    ours = np.array([O.round_bf16(x) for x in O.act(O.SILU, gf[ok].astype(np.float64))])
    mism = np.sum(eager != ours)
    assert mism <= 10, mism


def test_nvfp4_backward_is_nvfp4_of_the_backward_values():
    """NVFP4 backward: the [M, 2N] = [dGate | dUp] fp32 values quantised by
    the NVFP4 block rule (codes [M, N] packed, 128x4 scales of [M, 2N/16])."""
    rng = np.random.default_rng(6)
    M, N = 200, 48
    mk = lambda: (rng.standard_normal((M, N)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    g, u, d = mk(), mk(), mk()
    for act in (O.SILU, O.GELU_TANH):
        r = O.glu_bwd(g, u, d, act=act, fmt=O.NVFP4)
        f = np.ascontiguousarray(O.glu_bwd(g, u, d, act=act, fmt=O.FP32)["out"])
        q = np.zeros((M, N), np.uint8)
        s = np.zeros(256 * 8, np.uint8)
        O.lib().orc_nvfp4_matrix(O._ptr(f), M, 2 * N, O._ptr(q), O._ptr(s))
        assert np.array_equal(q, r["out"]) and np.array_equal(s, r["s_nvfp4"])



# ------------------------------------------- ReLU and identity gates --
# ReGLU (relu(g) = g for g > 0, else +0) and the bilinear GLU (act = identity):
# the gated activations beyond SiLU and GELU.  With bf16 operands their values
# are exact products, so the oracle is pinned against torch's own fp32 and
# autograd results bit for bit, and against the other activations where
# they coincide.

def _bf16_f32(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32)


def test_relu_identity_vs_torch_float64():
    x = torch.linspace(-5, 5, 10001, dtype=torch.float64)
    x = torch.cat([x, torch.tensor([0.0, -0.0, 1e-300, -1e-300, 3e38, -3e38, math.inf, -math.inf, math.nan],
                                   dtype=torch.float64)])
    # NaN kept, as torch.relu keeps it
    assert np.array_equal(O.act(O.RELU, x.numpy()), torch.relu(x).numpy(), equal_nan=True)
    assert np.array_equal(O.act(O.IDENTITY, x.numpy()), x.numpy(), equal_nan=True)
    t = x.clone().requires_grad_(True)
    torch.relu(t).sum().backward()
    assert np.array_equal(O.act_grad(O.RELU, x.numpy()), t.grad.numpy())  # 1 at NaN: dY passes
    assert np.all(O.act_grad(O.IDENTITY, x.numpy()) == 1.0)
    # relu is +0 (not -0) at and below zero: h then takes the sign of up
    assert all(math.copysign(1, v) == 1 for v in O.act(O.RELU, [-2.0, -0.0, 0.0]))


def _spiky_inputs(M, N, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(3):
        v = rng.standard_normal((M, N)).astype(np.float32)
        v[rng.random((M, N)) < 0.01] = 60.0
        v[rng.random((M, N)) < 0.01] = 0.0
        out.append(_bf16_bits(v))
    return out


@pytest.mark.parametrize("kind", [O.RELU, O.IDENTITY])
def test_exact_product_activations_vs_torch(kind):
    # forward fp32 values are torch's fp32 relu(g) * u (exact products), the
    # backward ones torch's autograd of relu(g) * u * dY in float64, rounded
    g, u, d = _spiky_inputs(64, 96, 31 + kind)
    gf, uf, df = (torch.from_numpy(_bf16_f32(b)) for b in (g, u, d))
    fn = torch.relu if kind == O.RELU else (lambda t: t)
    h = O.glu_fwd(g, u, act=kind, fmt=O.FP32)["out"]
    assert np.array_equal(h, (fn(gf) * uf).numpy())
    gg = gf.double().requires_grad_(True)
    uu = uf.double().requires_grad_(True)
    (fn(gg) * uu * df.double()).sum().backward()
    ref = torch.cat([gg.grad, uu.grad], dim=1).float().numpy()
    assert np.array_equal(O.glu_bwd(g, u, d, act=kind, fmt=O.FP32)["out"], ref)


def test_relu_signed_zeros_hand_worked():
    # g = -1: relu = +0, so h = (+0) * up carries the sign of up; one MXFP8
    # block of such values has scale 0 and codes 0x00 / 0x80
    g = _bf16_bits(np.full((1, 32), -1.0))
    u = _bf16_bits(np.where(np.arange(32) % 2 == 0, 2.0, -2.0).reshape(1, 32))
    r = O.glu_fwd(g, u, act=O.RELU, fmt=O.MXFP8, mode=O.ROW)
    assert r["s_row"].tolist() == [[0]]
    assert r["q_row"][0].tolist() == [0x00, 0x80] * 16
    # backward, dY = 1: dGate = (dY * up) * 0 keeps the sign of up, dUp = dY * (+0) = +0
    d = _bf16_bits(np.ones((1, 32)))
    out = O.glu_bwd(g, u, d, act=O.RELU, fmt=O.FP32)["out"][0]
    assert [math.copysign(1, v) for v in out[:32]] == [1.0, -1.0] * 16
    assert all(v == 0 and math.copysign(1, v) == 1 for v in out[32:])
    # dY = -1 flips both
    d = _bf16_bits(-np.ones((1, 32)))
    out = O.glu_bwd(g, u, d, act=O.RELU, fmt=O.FP32)["out"][0]
    assert [math.copysign(1, v) for v in out[:32]] == [-1.0, 1.0] * 16
    assert all(math.copysign(1, v) == -1 for v in out[32:])


@pytest.mark.parametrize("fmt,mode", [(O.MXFP8, O.BOTH), (O.NVFP4, O.ROW), (O.BF16, O.ROW)],
                         ids=["mxfp8_both", "nvfp4", "bf16"])
def test_relu_equals_identity_on_positive_gates(fmt, mode):
    rng = np.random.default_rng(41)
    M, N = 64, 128
    g = _bf16_bits(np.abs(rng.standard_normal((M, N))) + 2.0 ** -8)
    u, d = _bf16_bits(rng.standard_normal((M, N))), _bf16_bits(rng.standard_normal((M, N)))
    a = O.glu_fwd(g, u, act=O.RELU, fmt=fmt, mode=mode)
    b = O.glu_fwd(g, u, act=O.IDENTITY, fmt=fmt, mode=mode)
    assert all(np.array_equal(a[k], b[k]) for k in a)
    a = O.glu_bwd(g, u, d, act=O.RELU, fmt=fmt, mode=mode)
    b = O.glu_bwd(g, u, d, act=O.IDENTITY, fmt=fmt, mode=mode)
    assert all(np.array_equal(a[k], b[k]) for k in a)


def test_all_activations_agree_at_gate_32():
    # act(32) = 32 and act'(32) = 1 after rounding to fp32 for all four
    # activations, so every output of every format coincides
    rng = np.random.default_rng(42)
    M, N = 64, 64
    g = _bf16_bits(np.full((M, N), 32.0))
    u, d = _bf16_bits(rng.standard_normal((M, N))), _bf16_bits(rng.standard_normal((M, N)))
    for fmt, mode in ((O.MXFP8, O.BOTH), (O.NVFP4, O.ROW), (O.FP32, O.ROW)):
        ref_f = O.glu_fwd(g, u, act=O.SILU, fmt=fmt, mode=mode)
        ref_b = O.glu_bwd(g, u, d, act=O.SILU, fmt=fmt, mode=mode)
        for kind in (O.GELU_TANH, O.RELU, O.IDENTITY):
            f = O.glu_fwd(g, u, act=kind, fmt=fmt, mode=mode)
            b = O.glu_bwd(g, u, d, act=kind, fmt=fmt, mode=mode)
            assert all(np.array_equal(f[k], ref_f[k]) for k in f), (kind, fmt)
            assert all(np.array_equal(b[k], ref_b[k]) for k in b), (kind, fmt)


def test_relu_bf16_steps_is_one_rounding():
    # relu(g) of a bf16 gate is already bf16, so the bf16-step value is the
    # bf16 rounding of the exact product
    g, u, _ = _spiky_inputs(32, 64, 43)
    h = O.glu_fwd(g, u, act=O.RELU | O.BF16_STEPS, fmt=O.FP32)["out"]
    ref = (torch.relu(torch.from_numpy(_bf16_f32(g))) * torch.from_numpy(_bf16_f32(u))).to(torch.bfloat16)
    assert np.array_equal(h, ref.float().numpy())


# ------------------------------------------------------------ GELU (erf) --
# x * Phi(x), the erf form of GELU: defined in the oracle ahead of a GPU path.

def test_gelu_erf_vs_mpmath():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60

    def f(x):
        return x * mpmath.ncdf(x)

    xs = _all_bf16_in(-30.0, 30.0)[::5]
    ours, ours_d = O.act(O.GELU_ERF, xs), O.act_grad(O.GELU_ERF, xs)
    for x, y, dy in zip(xs, ours, ours_d):
        X = mpmath.mpf(float(x))
        ref, dref = f(X), mpmath.ncdf(X) + X * mpmath.npdf(X)
        # erfc's relative condition number grows like x^2 in the negative tail
        cond = 1.0 + float(x) ** 2
        assert abs(y - float(ref)) <= 1e-15 * cond * abs(float(ref)) + 1e-300, (x, y, float(ref))
        scale = abs(float(mpmath.ncdf(X))) + abs(float(X * mpmath.npdf(X)))  # act' has a zero near -0.75
        assert abs(dy - float(dref)) <= 1e-15 * cond * scale + 1e-300, (x, dy, float(dref))


def test_gelu_erf_vs_torch_float64():
    # torch evaluates 0.5 x (1 + erf(x / sqrt 2)), which cancels for x << 0;
    # stay where that library form is itself accurate (the tail is pinned
    # against mpmath above)
    x = torch.linspace(-3, 20, 20001, dtype=torch.float64)
    assert np.allclose(O.act(O.GELU_ERF, x.numpy()), torch.nn.functional.gelu(x).numpy(), rtol=1e-12, atol=1e-300)
    t = x.clone().requires_grad_(True)
    torch.nn.functional.gelu(t).sum().backward()
    assert np.allclose(O.act_grad(O.GELU_ERF, x.numpy()), t.grad.numpy(), rtol=1e-12, atol=1e-15)


def test_gelu_erf_special_values_and_differences():
    assert O.act(O.GELU_ERF, [0.0])[0] == 0.0
    assert O.act_grad(O.GELU_ERF, [0.0])[0] == 0.5
    assert np.float32(O.act(O.GELU_ERF, [60.0])[0]) == np.float32(60.0)
    assert np.float32(O.act_grad(O.GELU_ERF, [60.0])[0]) == np.float32(1.0)
    assert math.copysign(1, O.act(O.GELU_ERF, [-30.0])[0]) == -1  # a tiny negative value, not 0
    assert math.copysign(1, O.act(O.GELU_ERF, [-40.0])[0]) == -1  # Phi underflows: -0
    xs = np.linspace(-9, 9, 1801)
    h = 1e-5
    fd = (O.act(O.GELU_ERF, xs + h) - O.act(O.GELU_ERF, xs - h)) / (2 * h)
    assert np.allclose(O.act_grad(O.GELU_ERF, xs), fd, rtol=0, atol=1e-8)
    # close to the tanh approximation it was built to approximate (|diff| < 5e-4)
    assert np.max(np.abs(O.act(O.GELU_ERF, xs) - O.act(O.GELU_TANH, xs))) < 5e-4


# ---- non-finite blocks ------------------------------------------------------
# The pages name the NaN/Inf regime without fixing its bytes, so the bytes
# the oracle writes are a reading.  What the format definitions do fix (OCP
# MX v1.0: the E8M0 byte 0xFF and the E4M3 bytes 0x7F/0xFF are NaN; E2M1 has
# no NaN) is checked here with ml_dtypes' decoders: a block whose fp32 values
# hold a NaN or an infinity decodes to NaN in every element, and every other
# block decodes to finite values.

def _nonfinite_inputs(M, N, seed):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((M, N)).astype(np.float32)
    u = rng.standard_normal((M, N)).astype(np.float32)
    d = rng.standard_normal((M, N)).astype(np.float32)
    for t in (g, u, d):
        for _ in range(6):  # scattered, so rows, columns and blocks differ
            t[rng.integers(M), rng.integers(N)] = rng.choice([np.nan, np.inf, -np.inf])
    return _bf16_bits(g), _bf16_bits(u), _bf16_bits(d)


def _blocks_nonfinite(h, along_rows, k):
    """[blocks] mask: does each k-element block of h hold a NaN or an Inf."""
    bad = ~np.isfinite(h)
    if not along_rows:
        bad = bad.T
    R, C = bad.shape
    return bad.reshape(R, C // k, k).any(axis=2)


def _check_decoded(deq_blocks, bad):
    assert bad.any() and (~bad).any()
    assert np.isnan(deq_blocks[bad]).all()
    assert np.isfinite(deq_blocks[~bad]).all()


@pytest.mark.parametrize("kind", [O.SILU, O.GELU_TANH, O.RELU, O.IDENTITY, O.GELU_ERF])
@pytest.mark.parametrize("direction", ["fwd", "bwd"])
def test_nonfinite_blocks_decode_to_nan_mxfp8(kind, direction):
    M, N = 64, 256
    g, u, d = _nonfinite_inputs(M, N, 40 + kind)
    if direction == "fwd":
        r = O.glu_fwd(g, u, act=kind, fmt=O.MXFP8, mode=O.BOTH, want_h=True)
    else:
        r = O.glu_bwd(g, u, d, act=kind, fmt=O.MXFP8, mode=O.BOTH, want_h=True)
    h = r["h"]
    e4m3 = lambda q: q.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    e8m0 = lambda s: s.view(ml_dtypes.float8_e8m0fnu).astype(np.float64)
    for along_rows, q, s in ((True, r["q_row"], r["s_row"]), (False, r["q_col"], r["s_col"])):
        R, C = q.shape
        deq = e4m3(q).reshape(R, C // 32, 32) * e8m0(s)[:, :, None]
        _check_decoded(deq, _blocks_nonfinite(h, along_rows, 32))


@pytest.mark.parametrize("kind", [O.SILU, O.GELU_TANH, O.RELU, O.IDENTITY, O.GELU_ERF])
@pytest.mark.parametrize("direction", ["fwd", "bwd"])
def test_nonfinite_blocks_decode_to_nan_nvfp4(kind, direction):
    M, N = 160, 128  # two 128-row tiles of the scale layout, the second ragged
    g, u, d = _nonfinite_inputs(M, N, 50 + kind)
    if direction == "fwd":
        r = O.glu_fwd(g, u, act=kind, fmt=O.NVFP4, want_h=True)
    else:
        r = O.glu_bwd(g, u, d, act=kind, fmt=O.NVFP4, want_h=True)
    h = r["h"]
    W = h.shape[1]
    codes = np.empty((M, W), np.uint8)
    codes[:, 0::2] = r["out"] & 0xF
    codes[:, 1::2] = r["out"] >> 4
    e2m1 = codes.view(ml_dtypes.float4_e2m1fn).astype(np.float64)
    cp = -(-(W // 16) // 4) * 4
    sb = np.array([[r["s_nvfp4"][O.swizzle_offset(i, j, cp)] for j in range(W // 16)] for i in range(M)],
                  np.uint8)
    deq = e2m1.reshape(M, W // 16, 16) * sb.view(ml_dtypes.float8_e4m3fn).astype(np.float64)[:, :, None]
    _check_decoded(deq, _blocks_nonfinite(h, True, 16))
