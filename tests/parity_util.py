"""Comparison of the CUDA path with the CPU oracle under the stated rules.

Rules (the target's correctness statement):
  * scales are bit-exact;
  * codes are bit-exact, except where the oracle's fp32 pre-quant value lies
    within 2 fp32 ulps of a code rounding boundary; there one code step (same
    sign, adjacent magnitude) is allowed, and such elements are counted;
  * unquantised fp32 output: max relative error 1e-5 against the oracle;
    bf16 output: equal, except within 2 fp32 ulps of a bf16 midpoint (one
    bf16 step allowed, counted).
Expected values always come from ``oracle`` on host copies of the very same
input bytes.
"""
from __future__ import annotations

import numpy as np

import oracle as O

WINDOW_ULPS = 2


# Counts over every comparison of the session (codes and scales compared,
# codes differing by one step inside the 2-ulp window), reported at the end
# of a pytest run (tests/conftest.py).
TOTALS = {"elements": 0, "scales": 0, "window_mismatch": 0}


class Stats(dict):
    def add(self, k, v):
        self[k] = self.get(k, 0) + int(v)
        tail = k.rsplit(".", 1)[-1]
        if tail in TOTALS:
            TOTALS[tail] += int(v)


def _adjacent_e4m3(a, b):
    return ((a & 0x80) == (b & 0x80)) & (np.abs((a & 0x7F).astype(np.int32) - (b & 0x7F).astype(np.int32)) == 1)


def _adjacent_e2m1(a, b):
    return ((a & 0x8) == (b & 0x8)) & (np.abs((a & 0x7).astype(np.int32) - (b & 0x7).astype(np.int32)) == 1)


def check_codes(q_gpu, q_ref, v_ref, fmt, stats: Stats, what: str):
    """Compare code arrays (unpacked, one code per element)."""
    bad = q_gpu != q_ref
    n = int(bad.sum())
    stats.add(f"{what}.elements", q_ref.size)
    if n == 0:
        return
    idx = np.nonzero(bad.ravel())[0]
    g, r, v = q_gpu.ravel()[idx], q_ref.ravel()[idx], v_ref.ravel()[idx]
    near = O.boundary_ulps(fmt, v) <= WINDOW_ULPS
    adj = _adjacent_e4m3(g, r) if fmt == O.MXFP8 else _adjacent_e2m1(g, r)
    ok = near & adj
    stats.add(f"{what}.window_mismatch", ok.sum())
    if not ok.all():
        j = np.nonzero(~ok)[0][0]
        raise AssertionError(
            f"{what}: {int((~ok).sum())} code mismatches outside the 2-ulp window "
            f"(first: gpu {g[j]:#04x} ref {r[j]:#04x} v {v[j]!r}); total mismatches {n}")


def check_scales(s_gpu, s_ref, stats: Stats, what: str):
    stats.add(f"{what}.scales", s_ref.size)
    bad = s_gpu != s_ref
    if bad.any():
        i = np.nonzero(bad.ravel())[0][0]
        raise AssertionError(f"{what}: {int(bad.sum())} scale mismatches "
                             f"(first at flat {i}: gpu {s_gpu.ravel()[i]} ref {s_ref.ravel()[i]})")


def mx_prequant_row(h, s_row):
    """v = h * 2^-e for rowwise blocks (exact in fp32)."""
    e = np.repeat(s_row.astype(np.int32), 32, axis=1) - 127
    return (h.astype(np.float64) * np.exp2(-e.astype(np.float64))).astype(np.float32)


def mx_prequant_col(h, s_col):
    """v in the [W, M] colwise layout."""
    e = np.repeat(s_col.astype(np.int32), 32, axis=1) - 127
    return (h.T.astype(np.float64) * np.exp2(-e.astype(np.float64))).astype(np.float32)


def check_mx(gpu: dict, ref: dict, mode: int, stats: Stats, what: str):
    h = ref["h"]
    if mode & O.ROW:
        check_scales(gpu["s_row"], ref["s_row"], stats, what + ".row")
        check_codes(gpu["q_row"], ref["q_row"], mx_prequant_row(h, ref["s_row"]), O.MXFP8, stats,
                    what + ".row")
    if mode & O.COL:
        check_scales(gpu["s_col"], ref["s_col"], stats, what + ".col")
        check_codes(gpu["q_col"], ref["q_col"], mx_prequant_col(h, ref["s_col"]), O.MXFP8, stats,
                    what + ".col")


def unswizzle(s_flat, M, N):
    """128x4 layout -> plain [M, N/16] scale matrix (padding dropped)."""
    C = N // 16
    cp = -(-C // 4) * 4
    r = np.arange(M)[:, None]
    c = np.arange(C)[None, :]
    off = ((r // 128) * (cp // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)
    return s_flat[off]


def check_nvfp4(gpu: dict, ref: dict, M: int, N: int, stats: Stats, what: str):
    # the whole padded scale buffer (padding must be zero on both sides)
    check_scales(gpu["s_row"], ref["s_nvfp4"], stats, what + ".scale_buffer")
    q_g, q_r = gpu["q_row"], ref["out"]
    unpack = lambda q: np.stack([q & 0xF, q >> 4], axis=-1).reshape(q.shape[0], -1)
    s = O.e4m3_decode(unswizzle(ref["s_nvfp4"], M, N)).astype(np.float32)
    sv = np.repeat(s, 16, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = np.where(sv == 0, 0, ref["h"] / np.where(sv == 0, 1, sv)).astype(np.float32)
    check_codes(unpack(q_g), unpack(q_r), v, O.NVFP4, stats, what + ".codes")


def check_plain(gpu_out, ref: dict, fmt: int, stats: Stats, what: str):
    h = ref["h"]
    if fmt == O.FP32:
        g = gpu_out.astype(np.float64)
        r = h.astype(np.float64)
        fin = np.isfinite(r)
        assert np.array_equal(np.isnan(gpu_out), np.isnan(h)), what + ": NaN pattern differs"
        assert np.array_equal(g[~fin & ~np.isnan(r)], r[~fin & ~np.isnan(r)]), what + ": Inf differs"
        rel = np.abs(g[fin] - r[fin]) / np.maximum(np.abs(r[fin]), np.finfo(np.float32).tiny)
        mx = float(rel.max()) if rel.size else 0.0
        stats["%s.max_rel" % what] = max(stats.get("%s.max_rel" % what, 0.0), mx)
        stats.add(what + ".ulp_diff", (gpu_out != h).sum())
        assert mx <= 1e-5, f"{what}: max relative error {mx}"
    else:
        ref_b = ref["out"]
        isnan = lambda b: ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)
        assert np.array_equal(isnan(gpu_out), isnan(ref_b)), what + ": bf16 NaN pattern differs"
        # NaN payloads are not part of the contract: any NaN equals any NaN
        bad = (gpu_out != ref_b) & ~isnan(ref_b)
        stats.add(what + ".elements", ref_b.size)
        if bad.any():
            hv = h[bad]
            near = O.boundary_ulps(O.BF16, hv) <= WINDOW_ULPS
            step = np.abs(gpu_out[bad].astype(np.int32) - ref_b[bad].astype(np.int32)) == 1
            ok = near & step
            stats.add(what + ".window_mismatch", ok.sum())
            assert ok.all(), f"{what}: {int((~ok).sum())} bf16 mismatches outside the window"


def host_bits(t):
    """bf16 tensor -> host uint16 numpy array."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t):
    import torch
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return host_bits(t)
    return t.detach().cpu().numpy()


# ---- full-size comparison with counts (pre-quant values only where needed) --

def _nvfp4_scale_offsets(r, c, W):
    """Byte offsets of scales (r, c) of a [*, W/16] NVFP4 scale matrix in the
    128x4 layout."""
    cp = -(-(W // 16) // 4) * 4
    return ((r // 128) * (cp // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)


def compare_counts(gpu: dict, ref: dict, fmt: int, mode: int, M: int, W: int, h_rows) -> dict:
    """Compare one call's outputs with the oracle's under the rules above and
    return counts instead of raising: compared elements and scales, scale
    mismatches (the rules allow none), code mismatches inside the 2-ulp
    window with one code step (allowed, counted) and outside it (none
    allowed).  The oracle's exact values are needed only where codes differ;
    ``h_rows(rows)`` returns them ([len(rows), W] fp32, the FP32-mode oracle
    on those rows), so a full-size call needs no [M, W] array of them."""
    res = {"elements": 0, "scales": 0, "scale_mismatches": 0, "code_mismatches": 0,
           "window": 0, "out_of_window": 0}

    def codes(q_g, q_r, to_rc, v_of, fmt_c):
        bad = np.flatnonzero(q_g.ravel() != q_r.ravel())
        res["elements"] += q_r.size
        if bad.size == 0:
            return
        res["code_mismatches"] += bad.size
        r, c = to_rc(bad)
        rows, inv = np.unique(r, return_inverse=True)
        h = np.asarray(h_rows(rows), np.float32)[inv, c]
        v = v_of(h, r, c)
        g, q = q_g.ravel()[bad], q_r.ravel()[bad]
        if fmt_c == BF16_CODES:
            isnan = lambda b: ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)
            nan_ok = isnan(g) & isnan(q)
            ok = nan_ok | ((O.boundary_ulps(O.BF16, v) <= WINDOW_ULPS)
                           & (np.abs(g.astype(np.int32) - q.astype(np.int32)) == 1))
        else:
            adj = _adjacent_e4m3(g, q) if fmt_c == O.MXFP8 else _adjacent_e2m1(g, q)
            ok = (O.boundary_ulps(fmt_c, v) <= WINDOW_ULPS) & adj
        res["window"] += int(ok.sum())
        res["out_of_window"] += int((~ok).sum())

    def scales(s_g, s_r):
        res["scales"] += s_r.size
        res["scale_mismatches"] += int(np.count_nonzero(s_g != s_r))

    if fmt in (O.MXFP8,):
        if mode & O.ROW:
            scales(gpu["s_row"], ref["s_row"])
            s = ref["s_row"].astype(np.int32)
            codes(gpu["q_row"], ref["q_row"], lambda i: (i // W, i % W),
                  lambda h, r, c: (h.astype(np.float64) * np.exp2(127.0 - s[r, c // 32])).astype(np.float32),
                  O.MXFP8)
        if mode & O.COL:
            scales(gpu["s_col"], ref["s_col"])
            s = ref["s_col"].astype(np.int32)
            codes(gpu["q_col"], ref["q_col"], lambda i: (i % M, i // M),
                  lambda h, r, c: (h.astype(np.float64) * np.exp2(127.0 - s[c, r // 32])).astype(np.float32),
                  O.MXFP8)
    elif fmt == O.NVFP4:
        scales(gpu["s_row"], ref["s_nvfp4"])
        unpack = lambda q: np.stack([q & 0xF, q >> 4], axis=-1).reshape(q.shape[0], -1)
        sb = ref["s_nvfp4"]

        def v_nv(h, r, c):
            s = O.e4m3_decode(sb[_nvfp4_scale_offsets(r, c // 16, W)]).astype(np.float32)
            with np.errstate(divide="ignore", invalid="ignore"):
                return np.where(s == 0, np.float32(0), h / np.where(s == 0, 1, s)).astype(np.float32)
        codes(unpack(gpu["q_row"]), unpack(ref["out"]), lambda i: (i // W, i % W), v_nv, O.NVFP4)
    elif fmt == O.BF16:
        codes(gpu["out"], ref["out"], lambda i: (i // W, i % W), lambda h, r, c: h, BF16_CODES)
    else:
        raise ValueError("compare_counts covers MXFP8, NVFP4 and BF16 outputs")
    res["ok"] = res["scale_mismatches"] == 0 and res["out_of_window"] == 0
    return res


BF16_CODES = -1  # compare_counts: the codes are bf16 bit patterns
