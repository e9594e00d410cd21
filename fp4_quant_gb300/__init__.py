"""fp4_quant_gb300 — fused gated-GLU + block-scaled quantisation on GB300.

A thin ctypes binding of the C ABI in ``include/glu_quant.h``
(``libglu_quant.so``, built in-tree by ``fp4_quant_gb300.build``).  The
functions with the C names take the C argument structs and a stream handle
and do nothing but marshal; every step of the computation runs in the CUDA
kernels.  ``fwd``/``bwd`` are conveniences that allocate the outputs with
torch on the inputs' device and fill the argument struct from tensors.

There is no CPU or eager fallback: if the library is missing, the first call
raises ImportError (importing the package alone does not, so that
``python -m fp4_quant_gb300.build`` can create it).
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "glu_quant_fwd", "glu_quant_bwd", "glu_quant_fwd_nvfp4_gs", "glu_quant_fwd_sizes", "glu_quant_bwd_sizes",
    "glu_quant_status_str", "glu_quant_abi_version", "glu_quant_device_errors",
    "glu_quant_gemm_fwd", "glu_quant_gemm_sizes", "GluQuantGemmArgs", "gemm",
    "GluQuantFwdArgs", "GluQuantBwdArgs",
    "GluQuantError", "fwd", "bwd", "library_path",
    "ACT_SILU", "ACT_GELU_TANH", "ACT_RELU", "ACT_IDENTITY", "ACT_GELU_ERF", "ACT_BF16_STEPS", "FMT_MXFP8", "FMT_NVFP4", "FMT_BF16", "FMT_FP32", "FMT_MXFP8_128X4",
    "MODE_ROW", "MODE_COL", "MODE_BOTH", "LAYOUT_SPLIT", "LAYOUT_INTERLEAVED",
]

ACT_SILU, ACT_GELU_TANH, ACT_RELU, ACT_IDENTITY, ACT_GELU_ERF = 0, 1, 2, 3, 4  # SiLU, GELU (tanh), ReLU (ReGLU), identity (bilinear), GELU (erf)
ACT_BF16_STEPS = 16  # OR-ed into act (forward): the eager bf16 values RN_bf16(RN_bf16(act(g)) * up)
FMT_MXFP8, FMT_NVFP4, FMT_BF16, FMT_FP32, FMT_MXFP8_128X4 = 0, 1, 2, 3, 4
MODE_ROW, MODE_COL, MODE_BOTH = 1, 2, 3
LAYOUT_SPLIT, LAYOUT_INTERLEAVED = 0, 1

GLU_OK, GLU_EINVAL, GLU_ESHAPE, GLU_EALIGN, GLU_EDEVICE, GLU_ELAUNCH = 0, -1, -2, -3, -4, -5

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libglu_quant.so")


def library_path() -> str:
    return _LIB_PATH


class GluQuantFwdArgs(ctypes.Structure):
    """Mirror of ``glu_quant_fwd_args``."""
    _fields_ = [("act", ctypes.c_int32), ("fmt", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("layout", ctypes.c_int32),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("ld_in", ctypes.c_int64),
                ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p),
                ("q_row", ctypes.c_void_p), ("s_row", ctypes.c_void_p),
                ("q_col", ctypes.c_void_p), ("s_col", ctypes.c_void_p),
                ("out", ctypes.c_void_p)]


class GluQuantBwdArgs(ctypes.Structure):
    """Mirror of ``glu_quant_bwd_args``."""
    _fields_ = [("act", ctypes.c_int32), ("fmt", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("layout", ctypes.c_int32),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("ld_in", ctypes.c_int64),
                ("ld_dy", ctypes.c_int64),
                ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("dy", ctypes.c_void_p),
                ("q_row", ctypes.c_void_p), ("s_row", ctypes.c_void_p),
                ("q_col", ctypes.c_void_p), ("s_col", ctypes.c_void_p),
                ("out", ctypes.c_void_p)]


class GluQuantGemmArgs(ctypes.Structure):
    """Mirror of ``glu_quant_gemm_args``."""
    _fields_ = [("act", ctypes.c_int32), ("fmt", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("M", ctypes.c_int64), ("H", ctypes.c_int64), ("K", ctypes.c_int64),
                ("ld_x", ctypes.c_int64), ("ld_w", ctypes.c_int64),
                ("x", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("q", ctypes.c_void_p), ("s", ctypes.c_void_p)]


class GluQuantError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({glu_quant_status_str(status)})")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it with `python -m fp4_quant_gb300.build` "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(_LIB_PATH)
    lib.glu_quant_fwd.argtypes = [ctypes.POINTER(GluQuantFwdArgs), ctypes.c_void_p]
    lib.glu_quant_fwd.restype = ctypes.c_int
    lib.glu_quant_fwd_nvfp4_gs.argtypes = [ctypes.POINTER(GluQuantFwdArgs), ctypes.c_void_p, ctypes.c_void_p]
    lib.glu_quant_fwd_nvfp4_gs.restype = ctypes.c_int
    lib.glu_quant_bwd.argtypes = [ctypes.POINTER(GluQuantBwdArgs), ctypes.c_void_p]
    lib.glu_quant_bwd.restype = ctypes.c_int
    lib.glu_quant_fwd_sizes.argtypes = [ctypes.POINTER(GluQuantFwdArgs), ctypes.POINTER(ctypes.c_size_t)]
    lib.glu_quant_fwd_sizes.restype = ctypes.c_int
    lib.glu_quant_bwd_sizes.argtypes = [ctypes.POINTER(GluQuantBwdArgs), ctypes.POINTER(ctypes.c_size_t)]
    lib.glu_quant_bwd_sizes.restype = ctypes.c_int
    lib.glu_quant_status_str.argtypes = [ctypes.c_int]
    lib.glu_quant_status_str.restype = ctypes.c_char_p
    lib.glu_quant_abi_version.argtypes = []
    lib.glu_quant_abi_version.restype = ctypes.c_int
    lib.glu_quant_gemm_fwd.argtypes = [ctypes.POINTER(GluQuantGemmArgs), ctypes.c_void_p]
    lib.glu_quant_gemm_fwd.restype = ctypes.c_int
    lib.glu_quant_gemm_sizes.argtypes = [ctypes.POINTER(GluQuantGemmArgs), ctypes.POINTER(ctypes.c_size_t)]
    lib.glu_quant_gemm_sizes.restype = ctypes.c_int
    lib.glu_quant_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32),
                                            ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
    lib.glu_quant_device_errors.restype = ctypes.c_int
    return lib


_handle = None


def _lib() -> ctypes.CDLL:
    global _handle
    if _handle is None:
        _handle = _load()
    return _handle


# ---- the C entry points, same names -----------------------------------------

def glu_quant_fwd(args: GluQuantFwdArgs, stream: int | None) -> int:
    return _lib().glu_quant_fwd(ctypes.byref(args), stream)


def glu_quant_fwd_nvfp4_gs(args: GluQuantFwdArgs, amax: int | None, stream: int | None) -> int:
    return _lib().glu_quant_fwd_nvfp4_gs(ctypes.byref(args), amax, stream)


def glu_quant_bwd(args: GluQuantBwdArgs, stream: int | None) -> int:
    return _lib().glu_quant_bwd(ctypes.byref(args), stream)


def glu_quant_fwd_sizes(args: GluQuantFwdArgs) -> tuple[int, tuple[int, int, int, int]]:
    s = (ctypes.c_size_t * 4)()
    st = _lib().glu_quant_fwd_sizes(ctypes.byref(args), s)
    return st, tuple(s)


def glu_quant_bwd_sizes(args: GluQuantBwdArgs) -> tuple[int, tuple[int, int, int, int]]:
    s = (ctypes.c_size_t * 4)()
    st = _lib().glu_quant_bwd_sizes(ctypes.byref(args), s)
    return st, tuple(s)


def glu_quant_gemm_fwd(args: GluQuantGemmArgs, stream: int | None) -> int:
    return _lib().glu_quant_gemm_fwd(ctypes.byref(args), stream)


def glu_quant_gemm_sizes(args: GluQuantGemmArgs) -> tuple[int, tuple[int, int]]:
    s = (ctypes.c_size_t * 2)()
    st = _lib().glu_quant_gemm_sizes(ctypes.byref(args), s)
    return st, tuple(s)


def glu_quant_status_str(status: int) -> str:
    return _lib().glu_quant_status_str(status).decode()


def glu_quant_abi_version() -> int:
    return _lib().glu_quant_abi_version()


def glu_quant_device_errors(clear: bool = False) -> tuple[int, int, int]:
    """(status, forward error bits, backward error bits)."""
    f, b = ctypes.c_uint32(0), ctypes.c_uint32(0)
    st = _lib().glu_quant_device_errors(ctypes.byref(f), ctypes.byref(b), int(clear))
    return st, f.value, b.value


# ---- tensor conveniences ------------------------------------------------------

def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(device):
    import torch
    return torch.cuda.current_stream(device).cuda_stream


def _out_tensors(fmt, mode, M, W, device):
    import torch
    u8 = torch.uint8
    e = torch.empty
    if fmt == FMT_MXFP8:
        return {"q_row": e((M, W), dtype=u8, device=device) if mode & MODE_ROW else None,
                "s_row": e((M, W // 32), dtype=u8, device=device) if mode & MODE_ROW else None,
                "q_col": e((W, M), dtype=u8, device=device) if mode & MODE_COL else None,
                "s_col": e((W, M // 32), dtype=u8, device=device) if mode & MODE_COL else None,
                "out": None}
    if fmt == FMT_MXFP8_128X4:
        # scale matrices [M, W/32] and [W, M/32] in the padded 128x4 layout
        def sw(r, c):
            return (-(-r // 128) * 128) * (-(-c // 4) * 4)
        return {"q_row": e((M, W), dtype=u8, device=device) if mode & MODE_ROW else None,
                "s_row": e((sw(M, W // 32),), dtype=u8, device=device) if mode & MODE_ROW else None,
                "q_col": e((W, M), dtype=u8, device=device) if mode & MODE_COL else None,
                "s_col": e((sw(W, M // 32),), dtype=u8, device=device) if mode & MODE_COL else None,
                "out": None}
    if fmt == FMT_NVFP4:
        rp, cp = -(-M // 128) * 128, -(-W // 64) * 4
        return {"q_row": e((M, W // 2), dtype=u8, device=device),
                "s_row": e((rp * cp,), dtype=u8, device=device),
                "q_col": None, "s_col": None, "out": None}
    dt = torch.bfloat16 if fmt == FMT_BF16 else torch.float32
    return {"q_row": None, "s_row": None, "q_col": None, "s_col": None,
            "out": e((M, W), dtype=dt, device=device)}


def _check_input(t, name):
    import torch
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with unit column stride")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, but the current device is cuda:"
                         f"{torch.cuda.current_device()} (the kernels run on the current device)")


def _check_operands(M, N, layout, gate, up, dy=None):
    """The C layer sees only pointers and strides: check here that the
    tensors hold the rows and columns the arguments describe."""
    need = N if layout == LAYOUT_SPLIT else 2 * N
    if N <= 0 or gate.shape[1] < need:
        raise ValueError(f"gate has {gate.shape[1]} columns; N = {N} needs at least {need}")
    if layout == LAYOUT_SPLIT:
        if up is None:
            raise ValueError("the split layout needs `up`")
        if tuple(up.shape) != tuple(gate.shape):
            raise ValueError(f"up {tuple(up.shape)} and gate {tuple(gate.shape)} differ in shape")
    elif up is not None:
        raise ValueError("the interleaved layout takes gate = X and up = None")
    if dy is not None and (dy.shape[0] != M or dy.shape[1] < N):
        raise ValueError(f"dy {tuple(dy.shape)} does not hold [{M}, {N}]")


_OUT_KEYS = ("q_row", "s_row", "q_col", "s_col")


def _check_outputs(o, fmt, sizes, device):
    """Every output the call writes must exist, be a contiguous CUDA tensor
    on the inputs' device, have the format's dtype and hold the byte size
    the library reports (glu_quant_*_sizes); disabled outputs must be None."""
    import torch
    want = {"out": sizes[0]} if fmt in (FMT_BF16, FMT_FP32) else dict(zip(_OUT_KEYS, sizes))
    for k in ("q_row", "s_row", "q_col", "s_col", "out"):
        t = o.get(k)
        n = want.get(k, 0)
        if n == 0:
            if t is not None:
                raise ValueError(f"output {k} is not produced by this call; pass None")
            continue
        if t is None:
            raise ValueError(f"output {k} is required ({n} bytes)")
        dt = (torch.bfloat16 if fmt == FMT_BF16 else torch.float32) if k == "out" else torch.uint8
        if t.dtype != dt:
            raise TypeError(f"output {k} must be {dt}, got {t.dtype}")
        if not t.is_cuda or t.device != device:
            raise ValueError(f"output {k} must be on {device}, got {t.device}")
        if not t.is_contiguous():
            raise ValueError(f"output {k} must be contiguous")
        if t.numel() * t.element_size() < n:
            raise ValueError(f"output {k} holds {t.numel() * t.element_size()} bytes, needs {n}")


def fwd(gate, up=None, *, act=ACT_SILU, fmt=FMT_MXFP8, mode=MODE_ROW,
        layout=LAYOUT_SPLIT, N=None, out=None, stream=None, amax=None) -> dict:
    """Forward.  ``gate``/``up``: bf16 [M, N] (split) or ``gate`` = X [M, 2N]
    (interleaved, ``up`` None).  Returns the output dict (q_row, s_row,
    q_col, s_col, out); disabled outputs are None.  ``amax`` (NVFP4 only): a
    one-element fp32 CUDA tensor holding the tensor amax for the global
    scale (``glu_quant_fwd_nvfp4_gs``).  Raises GluQuantError on a nonzero
    status (nothing was launched then)."""
    _check_input(gate, "gate")
    if up is not None:
        _check_input(up, "up")
        if up.stride(0) != gate.stride(0):
            raise ValueError("gate and up must share the row stride")
    M = gate.shape[0]
    if N is None:
        N = gate.shape[1] if layout == LAYOUT_SPLIT else gate.shape[1] // 2
    _check_operands(M, N, layout, gate, up)
    o = out if out is not None else _out_tensors(fmt, mode, M, N, gate.device)
    a = GluQuantFwdArgs(act, fmt, mode, layout, M, N, gate.stride(0), _ptr(gate), _ptr(up),
                        _ptr(o.get("q_row")), _ptr(o.get("s_row")), _ptr(o.get("q_col")),
                        _ptr(o.get("s_col")), _ptr(o.get("out")))
    st, sizes = glu_quant_fwd_sizes(a)
    if st != GLU_OK:
        raise GluQuantError(st, "glu_quant_fwd_sizes")
    _check_outputs(o, fmt, sizes, gate.device)
    sh = stream if stream is not None else _stream_handle(gate.device)
    if amax is not None:
        import torch
        if amax.dtype != torch.float32 or amax.numel() < 1 or amax.device != gate.device:
            raise ValueError("amax must be a float32 tensor of at least one element on the inputs' device")
        st = glu_quant_fwd_nvfp4_gs(a, _ptr(amax), sh)
        if st != GLU_OK:
            raise GluQuantError(st, "glu_quant_fwd_nvfp4_gs")
        return o
    st = glu_quant_fwd(a, sh)
    if st != GLU_OK:
        raise GluQuantError(st, "glu_quant_fwd")
    return o


def bwd(gate, up, dy, *, act=ACT_SILU, fmt=FMT_MXFP8, mode=MODE_ROW,
        layout=LAYOUT_SPLIT, N=None, out=None, stream=None) -> dict:
    """Backward: outputs of the logical [M, 2N] matrix [dGate | dUp]."""
    _check_input(gate, "gate")
    _check_input(dy, "dy")
    if up is not None:
        _check_input(up, "up")
        if up.stride(0) != gate.stride(0):
            raise ValueError("gate and up must share the row stride")
    M = gate.shape[0]
    if N is None:
        N = gate.shape[1] if layout == LAYOUT_SPLIT else gate.shape[1] // 2
    _check_operands(M, N, layout, gate, up, dy)
    o = out if out is not None else _out_tensors(fmt, mode, M, 2 * N, gate.device)
    a = GluQuantBwdArgs(act, fmt, mode, layout, M, N, gate.stride(0), dy.stride(0), _ptr(gate),
                        _ptr(up), _ptr(dy), _ptr(o.get("q_row")), _ptr(o.get("s_row")),
                        _ptr(o.get("q_col")), _ptr(o.get("s_col")), _ptr(o.get("out")))
    st, sizes = glu_quant_bwd_sizes(a)
    if st != GLU_OK:
        raise GluQuantError(st, "glu_quant_bwd_sizes")
    _check_outputs(o, fmt, sizes, gate.device)
    st = glu_quant_bwd(a, stream if stream is not None else _stream_handle(gate.device))
    if st != GLU_OK:
        raise GluQuantError(st, "glu_quant_bwd")
    return o


def gemm(x, w, *, act=ACT_GELU_TANH, fmt=FMT_NVFP4, layout=LAYOUT_INTERLEAVED, out=None,
         stream=None) -> dict:
    """The gate/up GEMM with the quantiser in its epilogue: ``x`` bf16
    [M, K], ``w`` bf16 [2H, K] (gate/up rows interleaved or split); returns
    {"q", "s"} (allocated unless ``out`` is given).  Raises GluQuantError on
    a nonzero status (nothing was launched then)."""
    import torch
    _check_input(x, "x")
    _check_input(w, "w")
    M, K = x.shape
    if w.shape[1] != K or w.shape[0] % 2 != 0:
        raise ValueError(f"w {tuple(w.shape)} does not hold [2H, {K}]")
    H = w.shape[0] // 2
    a = GluQuantGemmArgs(act, fmt, layout, 0, M, H, K, x.stride(0), w.stride(0), _ptr(x), _ptr(w),
                         None, None)
    st, sizes = glu_quant_gemm_sizes(a)
    if st != GLU_OK:
        raise GluQuantError(st, "glu_quant_gemm_sizes")
    if out is None:
        out = {"q": torch.empty(sizes[0], dtype=torch.uint8, device=x.device),
               "s": torch.empty(sizes[1], dtype=torch.uint8, device=x.device)}
    for k, n in zip(("q", "s"), sizes):
        t = out.get(k)
        if t is None or t.dtype != torch.uint8 or t.device != x.device or not t.is_contiguous() \
                or t.numel() < n:
            raise ValueError(f"output {k} must be a contiguous uint8 tensor of >= {n} bytes on {x.device}")
    a.q, a.s = _ptr(out["q"]), _ptr(out["s"])
    st = glu_quant_gemm_fwd(a, stream if stream is not None else _stream_handle(x.device))
    if st != GLU_OK:
        raise GluQuantError(st, "glu_quant_gemm_fwd")
    return out
