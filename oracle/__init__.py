"""Plain CPU oracle for the fused gated-GLU + block-scaled quantisation path.

TEST INFRASTRUCTURE ONLY.  The product (``fp4_quant_gb300``) never imports,
loads or calls this package; only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline legs of ``bench.py`` do.  The arithmetic lives in
``oracle.c`` (plain C, double-precision activations, bit-level encoders);
this module builds it with gcc and marshals numpy arrays to it with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

SILU, GELU_TANH, RELU, IDENTITY, GELU_ERF = 0, 1, 2, 3, 4
BF16_STEPS = 16  # OR-ed into act (forward): h = RN_bf16(RN_bf16(act(g)) * u)
MXFP8, NVFP4, BF16, FP32, MXFP8_128X4 = 0, 1, 2, 3, 4
ROW, COL, BOTH = 1, 2, 3
SPLIT, INTERLEAVED = 0, 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so (plain C11, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", "-fno-fast-math", "-Wall", _SRC, "-lm",
               "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class FwdArgs(ctypes.Structure):
    _fields_ = [("act", ctypes.c_int32), ("fmt", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("layout", ctypes.c_int32),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("ld_in", ctypes.c_int64),
                ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p),
                ("q_row", ctypes.c_void_p), ("s_row", ctypes.c_void_p),
                ("q_col", ctypes.c_void_p), ("s_col", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("s_nvfp4", ctypes.c_void_p),
                ("h", ctypes.c_void_p)]


class GemmArgs(ctypes.Structure):
    _fields_ = [("act", ctypes.c_int32), ("fmt", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("M", ctypes.c_int64), ("H", ctypes.c_int64), ("K", ctypes.c_int64),
                ("ld_x", ctypes.c_int64), ("ld_w", ctypes.c_int64),
                ("x", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("q", ctypes.c_void_p), ("s", ctypes.c_void_p),
                ("c", ctypes.c_void_p), ("h", ctypes.c_void_p)]


class BwdArgs(ctypes.Structure):
    _fields_ = [("act", ctypes.c_int32), ("fmt", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("layout", ctypes.c_int32),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("ld_in", ctypes.c_int64),
                ("ld_dy", ctypes.c_int64),
                ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("dy", ctypes.c_void_p),
                ("q_row", ctypes.c_void_p), ("s_row", ctypes.c_void_p),
                ("q_col", ctypes.c_void_p), ("s_col", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("h", ctypes.c_void_p)]


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            l = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            for name in ("orc_e4m3_encode_n", "orc_e2m1_encode_n", "orc_e8m0_rceil_n",
                         "orc_nvfp4_scale_n", "orc_bf16_rne_n"):
                getattr(l, name).argtypes = [P, P, i64]
                getattr(l, name).restype = None
            for name in ("orc_act_n", "orc_act_grad_n", "orc_boundary_ulps_n"):
                getattr(l, name).argtypes = [ctypes.c_int, P, P, i64]
                getattr(l, name).restype = None
            l.orc_encode_bits.argtypes = [ctypes.c_int, ctypes.c_uint32, i64, P, ctypes.c_int]
            l.orc_encode_bits.restype = None
            l.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            l.orc_e4m3_decode.restype = ctypes.c_float
            l.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
            l.orc_e2m1_decode.restype = ctypes.c_float
            l.orc_e8m0_decode.argtypes = [ctypes.c_uint8]
            l.orc_e8m0_decode.restype = ctypes.c_float
            l.orc_swizzle_offset.argtypes = [i64, i64, i64]
            l.orc_swizzle_offset.restype = i64
            l.orc_round_bf16.argtypes = [ctypes.c_double]
            l.orc_round_bf16.restype = ctypes.c_double
            l.orc_scales_128x4.argtypes = [ctypes.c_void_p, i64, i64, ctypes.c_void_p]
            l.orc_scales_128x4.restype = None
            l.orc_nvfp4_matrix.argtypes = [ctypes.c_void_p, i64, i64, ctypes.c_void_p, ctypes.c_void_p]
            l.orc_nvfp4_matrix.restype = None
            l.orc_glu_fwd.argtypes = [ctypes.POINTER(FwdArgs), ctypes.c_int]
            l.orc_glu_fwd.restype = ctypes.c_int
            l.orc_glu_bwd.argtypes = [ctypes.POINTER(BwdArgs), ctypes.c_int]
            l.orc_glu_bwd.restype = ctypes.c_int
            l.orc_gemm_glu_fwd.argtypes = [ctypes.POINTER(GemmArgs), ctypes.c_int]
            l.orc_gemm_glu_fwd.restype = ctypes.c_int
            _lib = l
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


# ---- scalar building blocks, vectorised ------------------------------------

def e4m3_encode(v) -> np.ndarray:
    v = _f32(v)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_n(_ptr(v), _ptr(out), v.size)
    return out


def e2m1_encode(v) -> np.ndarray:
    v = _f32(v)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e2m1_encode_n(_ptr(v), _ptr(out), v.size)
    return out


def e8m0_rceil(amax) -> np.ndarray:
    v = _f32(amax)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e8m0_rceil_n(_ptr(v), _ptr(out), v.size)
    return out


def nvfp4_scale(amax) -> np.ndarray:
    v = _f32(amax)
    out = np.empty(v.shape, np.uint8)
    lib().orc_nvfp4_scale_n(_ptr(v), _ptr(out), v.size)
    return out


def bf16_rne(v) -> np.ndarray:
    v = _f32(v)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_rne_n(_ptr(v), _ptr(out), v.size)
    return out


def e4m3_decode(c) -> np.ndarray:
    table = np.array([lib().orc_e4m3_decode(i) for i in range(256)], np.float32)
    return table[np.asarray(c, np.uint8)]


def e2m1_decode(c) -> np.ndarray:
    table = np.array([lib().orc_e2m1_decode(i) for i in range(16)], np.float32)
    return table[np.asarray(c, np.uint8)]


def e8m0_decode(s) -> np.ndarray:
    table = np.array([lib().orc_e8m0_decode(i) for i in range(256)], np.float32)
    return table[np.asarray(s, np.uint8)]


def act(kind: int, x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, np.float64))
    out = np.empty(x.shape, np.float64)
    lib().orc_act_n(kind, _ptr(x), _ptr(out), x.size)
    return out


def act_grad(kind: int, x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, np.float64))
    out = np.empty(x.shape, np.float64)
    lib().orc_act_grad_n(kind, _ptr(x), _ptr(out), x.size)
    return out


def boundary_ulps(fmt: int, v) -> np.ndarray:
    v = _f32(v)
    out = np.empty(v.shape, np.int64)
    lib().orc_boundary_ulps_n(fmt, _ptr(v), _ptr(out), v.size)
    return out


def encode_bits(kind: int, first: int, n: int, nthreads: int | None = None) -> np.ndarray:
    """Codes of the fp32 values with bit patterns first .. first+n-1
    (kind 0 = E4M3, 1 = E2M1)."""
    out = np.empty(n, np.uint8)
    lib().orc_encode_bits(kind, first, n, _ptr(out), nthreads or os.cpu_count() or 1)
    return out


def swizzle_offset(r: int, c: int, scale_cols_padded: int) -> int:
    return lib().orc_swizzle_offset(r, c, scale_cols_padded)


def scales_128x4(S: np.ndarray) -> np.ndarray:
    """A row-major scale matrix [R, C] in the padded 128x4 layout (flat)."""
    S = np.ascontiguousarray(S, dtype=np.uint8)
    R, C = S.shape
    out = np.empty((-(-R // 128) * 128) * (-(-C // 4) * 4), np.uint8)
    lib().orc_scales_128x4(_ptr(S), R, C, _ptr(out))
    return out


def round_bf16(x: float) -> float:
    """The nearest bf16 value of a double (ties to even), as a double."""
    return lib().orc_round_bf16(float(x))


def nvfp4_global_scale(amax: float) -> np.float32:
    """The global encode scale G = 2688 / amax in fp32 (IEEE division);
    1 for a zero, negative or non-finite amax."""
    a = np.float32(amax)
    if not (np.isfinite(a) and a > 0):
        return np.float32(1.0)
    return np.float32(np.float32(2688.0) / a)


def glu_fwd_nvfp4_gs(gate, up=None, *, act: int, amax: float, layout: int = SPLIT,
                     N: int | None = None, nthreads: int | None = None) -> dict:
    """NVFP4 with a global scale: v = RN_fp32(h * G), h the path's exact fp32
    values, then the unit-global-scale NVFP4 rule on v.  Returns out (codes),
    s_nvfp4 (padded 128x4 scales), h and v."""
    h = glu_fwd(gate, up, act=act, fmt=FP32, layout=layout, N=N, nthreads=nthreads)["out"]
    v = np.ascontiguousarray((h * nvfp4_global_scale(amax)).astype(np.float32))
    M, W = v.shape
    q = np.zeros((M, W // 2), np.uint8)
    s = np.zeros((-(-M // 128) * 128) * (-(-(W // 16) // 4) * 4), np.uint8)
    lib().orc_nvfp4_matrix(_ptr(v), M, W, _ptr(q), _ptr(s))
    return {"out": q, "s_nvfp4": s, "h": h, "v": v}


def _mx_128x4(res: dict) -> dict:
    """MXFP8_128X4 results from plain MXFP8 ones: the same codes, the scale
    matrices re-laid in the 128x4 layout."""
    for k in ("s_row", "s_col"):
        if res.get(k) is not None:
            res[k] = scales_128x4(res[k])
    return res


# ---- the path ---------------------------------------------------------------

def _bits(x: np.ndarray) -> np.ndarray:
    """bf16 data as uint16 bit patterns (accepts uint16 or ml_dtypes bf16)."""
    x = np.asarray(x)
    if x.dtype != np.uint16:
        x = x.view(np.uint16)
    return x


def out_shapes_fwd(fmt, mode, M, N):
    """Shapes of (q_row, s_row, q_col, s_col) or (codes, scales) or (out,)."""
    if fmt == MXFP8:
        return {"q_row": (M, N) if mode & ROW else None,
                "s_row": (M, N // 32) if mode & ROW else None,
                "q_col": (N, M) if mode & COL else None,
                "s_col": (N, M // 32) if mode & COL else None}
    if fmt == NVFP4:
        rp = -(-M // 128) * 128
        cp = -(-(N // 16) // 4) * 4
        return {"out": (M, N // 2), "s_nvfp4": (rp * cp,)}
    return {"out": (M, N)}


def glu_fwd(gate, up=None, *, act: int, fmt: int, mode: int = ROW,
            layout: int = SPLIT, N: int | None = None, want_h: bool = False,
            nthreads: int | None = None) -> dict:
    """Run the oracle forward.  ``gate`` is [M, ld] bf16 bits; for the
    interleaved layout ``gate`` is X [M, >=2N] and ``up`` is None."""
    if fmt == MXFP8_128X4:
        return _mx_128x4(glu_fwd(gate, up, act=act, fmt=MXFP8, mode=mode, layout=layout, N=N,
                                 want_h=want_h, nthreads=nthreads))
    g = np.ascontiguousarray(_bits(gate))
    u = None if up is None else np.ascontiguousarray(_bits(up))
    M, ld = g.shape
    if N is None:
        N = ld if layout == SPLIT else ld // 2
    if u is not None and u.shape != g.shape:
        raise ValueError("gate and up must have the same shape")
    res = {}
    for k, shp in out_shapes_fwd(fmt, mode, M, N).items():
        if shp is None:
            res[k] = None
        elif k == "out":
            dt = {BF16: np.uint16, FP32: np.float32, NVFP4: np.uint8}[fmt]
            res[k] = np.zeros(shp, dt)
        else:
            res[k] = np.zeros(shp, np.uint8)
    h = np.zeros((M, N), np.float32) if want_h else None
    a = FwdArgs(act, fmt, mode, layout, M, N, ld, _ptr(g).value,
                None if u is None else _ptr(u).value,
                *(None if res.get(k) is None else _ptr(res[k]).value
                  for k in ("q_row", "s_row", "q_col", "s_col", "out", "s_nvfp4")),
                None if h is None else _ptr(h).value)
    rc = lib().orc_glu_fwd(ctypes.byref(a), nthreads or os.cpu_count() or 1)
    if rc != 0:
        raise ValueError("oracle rejected the forward arguments")
    if want_h:
        res["h"] = h
    return res


def glu_bwd(gate, up, dy, *, act: int, fmt: int, mode: int = ROW,
            layout: int = SPLIT, N: int | None = None, want_h: bool = False,
            nthreads: int | None = None) -> dict:
    """Run the oracle backward: logical output [M, 2N] = [dGate | dUp]."""
    if fmt == MXFP8_128X4:
        return _mx_128x4(glu_bwd(gate, up, dy, act=act, fmt=MXFP8, mode=mode, layout=layout, N=N,
                                 want_h=want_h, nthreads=nthreads))
    g = np.ascontiguousarray(_bits(gate))
    u = None if up is None else np.ascontiguousarray(_bits(up))
    d = np.ascontiguousarray(_bits(dy))
    M, ld = g.shape
    if N is None:
        N = ld if layout == SPLIT else ld // 2
    W = 2 * N
    res = {}
    for k, shp in out_shapes_fwd(fmt, mode, M, W).items():
        if shp is None:
            res[k] = None
        elif k == "out":
            res[k] = np.zeros(shp, {BF16: np.uint16, FP32: np.float32, NVFP4: np.uint8}[fmt])
        else:
            res[k] = np.zeros(shp, np.uint8)
    h = np.zeros((M, W), np.float32) if want_h else None
    keys = ("q_row", "s_nvfp4" if fmt == NVFP4 else "s_row", "q_col", "s_col", "out")
    a = BwdArgs(act, fmt, mode, layout, M, N, ld, d.shape[1], _ptr(g).value,
                None if u is None else _ptr(u).value, _ptr(d).value,
                *(None if res.get(k) is None else _ptr(res[k]).value for k in keys),
                None if h is None else _ptr(h).value)
    rc = lib().orc_glu_bwd(ctypes.byref(a), nthreads or os.cpu_count() or 1)
    if rc != 0:
        raise ValueError("oracle rejected the backward arguments")
    if want_h:
        res["h"] = h
    return res


def gemm_glu_fwd(x, w, *, act: int, fmt: int, layout: int = INTERLEAVED, want_c: bool = False,
                 want_h: bool = False, nthreads: int | None = None) -> dict:
    """Run the oracle of the gate/up GEMM path: ``x`` bf16 bits [M, K], ``w``
    bf16 bits [2H, K].  Returns q, s (NVFP4: packed codes and padded 128x4
    scales; MXFP8 and MXFP8_128X4: codes and the scales in that layout) and,
    when asked, the fp32 projection c [M, 2H] and h [M, H]."""
    if fmt == MXFP8_128X4:
        r = gemm_glu_fwd(x, w, act=act, fmt=MXFP8, layout=layout, want_c=want_c, want_h=want_h,
                         nthreads=nthreads)
        r["s"] = scales_128x4(r["s"])
        return r
    xb = np.ascontiguousarray(_bits(x))
    wb = np.ascontiguousarray(_bits(w))
    M, K = xb.shape
    H = wb.shape[0] // 2
    if wb.shape[1] != K or wb.shape[0] != 2 * H:
        raise ValueError("w must be [2H, K]")
    if fmt == NVFP4:
        q = np.zeros((M, H // 2), np.uint8)
        s = np.zeros((-(-M // 128) * 128) * (-(-(H // 16) // 4) * 4), np.uint8)
    else:
        q = np.zeros((M, H), np.uint8)
        s = np.zeros((M, H // 32), np.uint8)
    c = np.zeros((M, 2 * H), np.float32) if want_c else None
    h = np.zeros((M, H), np.float32) if want_h else None
    a = GemmArgs(act, fmt, layout, 0, M, H, K, K, K, _ptr(xb).value, _ptr(wb).value,
                 _ptr(q).value, _ptr(s).value, None if c is None else _ptr(c).value,
                 None if h is None else _ptr(h).value)
    if lib().orc_gemm_glu_fwd(ctypes.byref(a), nthreads or os.cpu_count() or 1) != 0:
        raise ValueError("oracle rejected the GEMM arguments")
    res = {"q": q, "s": s}
    if want_c:
        res["c"] = c
    if want_h:
        res["h"] = h
    return res
