"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function ``include/glu_quant.h``
declares, and reject every bad argument with the documented status before
touching a device (argument checks run first, so on a machine without a GPU
a well-formed call reports GLU_EDEVICE and a malformed one its own error).
"""
import ctypes
import os
import re

import pytest

import fp4_quant_gb300 as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "glu_quant.h")
P = 1 << 12  # a 16-byte aligned placeholder address (never dereferenced)


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"GLU_API\s+[\w\s\*]+?\b(glu_quant_\w+)\s*\(", txt)))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert len(names) == 10, names
    lib = ctypes.CDLL(G.library_path())
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_status_strings():
    assert G.glu_quant_abi_version() == 5
    for st in (0, -1, -2, -3, -4, -5):
        assert G.glu_quant_status_str(st) != "unknown status"
    assert G.glu_quant_status_str(7) == "unknown status"


def fwd_args(**kw):
    a = dict(act=0, fmt=0, mode=1, layout=0, M=64, N=256, ld_in=256, gate=P, up=P,
             q_row=P, s_row=P, q_col=None, s_col=None, out=None)
    a.update(kw)
    return G.GluQuantFwdArgs(**a)


def bwd_args(**kw):
    a = dict(act=0, fmt=0, mode=1, layout=0, M=64, N=256, ld_in=256, ld_dy=256, gate=P, up=P,
             dy=P, q_row=P, s_row=P, q_col=None, s_col=None, out=None)
    a.update(kw)
    return G.GluQuantBwdArgs(**a)


def _no_gpu():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:
        return True


@pytest.mark.parametrize("kw,status", [
    (dict(act=5), G.GLU_EINVAL),
    (dict(act=21), G.GLU_EINVAL),
    (dict(act=32), G.GLU_EINVAL),
    (dict(fmt=5), G.GLU_EINVAL),
    (dict(mode=0), G.GLU_EINVAL),
    (dict(mode=4), G.GLU_EINVAL),
    (dict(layout=2), G.GLU_EINVAL),
    (dict(M=0), G.GLU_EINVAL),
    (dict(N=-32), G.GLU_EINVAL),
    (dict(gate=None), G.GLU_EINVAL),
    (dict(up=None), G.GLU_EINVAL),                         # split needs up
    (dict(layout=1, ld_in=512), G.GLU_EINVAL),              # interleaved must not pass up
    (dict(q_row=None), G.GLU_EINVAL),                      # enabled output missing
    (dict(q_col=P), G.GLU_EINVAL),                         # disabled output given
    (dict(out=P), G.GLU_EINVAL),
    (dict(fmt=1, mode=3), G.GLU_EINVAL),                   # NVFP4 is row only
    (dict(fmt=2, q_row=None, s_row=None, out=P, mode=2), G.GLU_EINVAL),
    (dict(N=240, ld_in=240), G.GLU_ESHAPE),                # N % 32 for MXFP8
    (dict(mode=2, q_row=None, s_row=None, q_col=P, s_col=P, M=40), G.GLU_ESHAPE),
    (dict(fmt=1, N=264, ld_in=264), G.GLU_ESHAPE),         # N % 16 for NVFP4
    (dict(ld_in=128), G.GLU_ESHAPE),                       # ld < N
    (dict(layout=1, up=None, ld_in=256), G.GLU_ESHAPE),    # interleaved ld < 2N
    (dict(M=1 << 62), G.GLU_ESHAPE),                       # size overflow
    (dict(M=1 << 31), G.GLU_ESHAPE),                       # 32-bit TMA row coordinates
    (dict(N=1 << 30, ld_in=1 << 30), G.GLU_ESHAPE),        # 2N columns of [dGate | dUp] / [2N, M]
    (dict(ld_in=260), G.GLU_EALIGN),                       # ld % 8
    (dict(gate=P + 2), G.GLU_EALIGN),
    (dict(s_row=P + 8), G.GLU_EALIGN),
])
def test_fwd_rejections(kw, status):
    assert G.glu_quant_fwd(fwd_args(**kw), None) == status


@pytest.mark.parametrize("kw,status", [
    (dict(act=16), G.GLU_EINVAL),                          # bf16 steps: forward only
    (dict(dy=None), G.GLU_EINVAL),
    (dict(fmt=1, mode=2, q_row=None, s_row=None, q_col=P, s_col=P), G.GLU_EINVAL),  # NVFP4 is row only
    (dict(ld_dy=128), G.GLU_ESHAPE),
    (dict(ld_dy=260), G.GLU_EALIGN),
    (dict(dy=P + 4), G.GLU_EALIGN),
    (dict(N=240, ld_in=240, ld_dy=240), G.GLU_ESHAPE),     # N % 32 (not 2N)
])
def test_bwd_rejections(kw, status):
    assert G.glu_quant_bwd(bwd_args(**kw), None) == status


def test_nvfp4_global_scale_rejections():
    nv = dict(fmt=1, layout=1, up=None, ld_in=512)
    assert G.glu_quant_fwd_nvfp4_gs(fwd_args(), P, None) == G.GLU_EINVAL        # not NVFP4
    assert G.glu_quant_fwd_nvfp4_gs(fwd_args(**nv), None, None) == G.GLU_EINVAL  # no amax
    assert G.glu_quant_fwd_nvfp4_gs(fwd_args(**nv), P + 2, None) == G.GLU_EALIGN
    assert G.glu_quant_fwd_nvfp4_gs(fwd_args(fmt=1, layout=1, up=None, ld_in=256), P, None) == G.GLU_ESHAPE


@pytest.mark.skipif(not _no_gpu(), reason="checks the no-device status")
def test_valid_call_without_device_reports_edevice():
    assert G.glu_quant_fwd(fwd_args(), None) == G.GLU_EDEVICE
    assert G.glu_quant_bwd(bwd_args(), None) == G.GLU_EDEVICE


def test_sizes():
    st, s = G.glu_quant_fwd_sizes(fwd_args(mode=3, q_col=P, s_col=P, M=4096, N=7168, ld_in=7168))
    assert st == 0 and s == (4096 * 7168, 4096 * 224, 7168 * 4096, 7168 * 128)
    st, s = G.glu_quant_bwd_sizes(bwd_args(mode=2, M=4096, N=7168, ld_in=7168, ld_dy=7168))
    assert st == 0 and s == (0, 0, 14336 * 4096, 14336 * 128)
    st, s = G.glu_quant_fwd_sizes(fwd_args(fmt=1, layout=1, M=784, N=16384, ld_in=32768))
    assert st == 0 and s == (784 * 8192, 896 * 1024, 0, 0)
    st, s = G.glu_quant_fwd_sizes(fwd_args(fmt=2, M=8, N=1001, ld_in=1008))
    assert st == 0 and s == (8 * 1001 * 2, 0, 0, 0)
    st, _ = G.glu_quant_fwd_sizes(fwd_args(N=250, ld_in=256))
    assert st == G.GLU_ESHAPE
    # MXFP8 with 128x4 scales: [R, C] padded to ceil(R/128)*128 x ceil(C/4)*4
    st, s = G.glu_quant_fwd_sizes(fwd_args(fmt=4, mode=3, q_col=P, s_col=P, M=160, N=800, ld_in=800))
    assert st == 0 and s == (160 * 800, 256 * 28, 800 * 160, 896 * 8)
    st, s = G.glu_quant_bwd_sizes(bwd_args(fmt=4, mode=1, M=96, N=416, ld_in=416, ld_dy=416))
    assert st == 0 and s == (96 * 832, 128 * 28, 0, 0)
    st, _ = G.glu_quant_fwd_sizes(fwd_args(fmt=5))
    assert st == G.GLU_EINVAL
    # NVFP4 backward: codes of [M, 2N] packed, scales of [M, 2N/16] in 128x4
    st, s = G.glu_quant_bwd_sizes(bwd_args(fmt=1, M=200, N=48, ld_in=48, ld_dy=48))
    assert st == 0 and s == (200 * 48, 256 * 8, 0, 0)


def test_binding_mirrors_the_header(tmp_path):
    """The ctypes structs and constants of the binding against the header as
    a C compiler sees it: struct sizes, every field offset, every enum and
    status value."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    fields = {"glu_quant_fwd_args": G.GluQuantFwdArgs, "glu_quant_bwd_args": G.GluQuantBwdArgs,
              "glu_quant_gemm_args": G.GluQuantGemmArgs}
    consts = {"GLU_ACT_SILU": G.ACT_SILU, "GLU_ACT_GELU_TANH": G.ACT_GELU_TANH, "GLU_ACT_RELU": G.ACT_RELU,
              "GLU_ACT_IDENTITY": G.ACT_IDENTITY, "GLU_ACT_GELU_ERF": G.ACT_GELU_ERF, "GLU_ACT_BF16_STEPS": G.ACT_BF16_STEPS,
              "GLU_FMT_MXFP8_E4M3": G.FMT_MXFP8, "GLU_FMT_NVFP4_E2M1": G.FMT_NVFP4, "GLU_FMT_BF16": G.FMT_BF16,
              "GLU_FMT_FP32": G.FMT_FP32, "GLU_FMT_MXFP8_E4M3_128X4": G.FMT_MXFP8_128X4,
              "GLU_MODE_ROW": G.MODE_ROW, "GLU_MODE_COL": G.MODE_COL, "GLU_MODE_BOTH": G.MODE_BOTH,
              "GLU_LAYOUT_SPLIT": G.LAYOUT_SPLIT, "GLU_LAYOUT_INTERLEAVED": G.LAYOUT_INTERLEAVED,
              "GLU_OK": G.GLU_OK, "GLU_EINVAL": G.GLU_EINVAL, "GLU_ESHAPE": G.GLU_ESHAPE,
              "GLU_EALIGN": G.GLU_EALIGN, "GLU_EDEVICE": G.GLU_EDEVICE, "GLU_ELAUNCH": G.GLU_ELAUNCH}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "glu_quant.h"', "int main(void) {"]
    for st, cls in fields.items():
        lines.append(f'  printf("size {st} %zu\\n", sizeof({st}));')
        for name, _ in cls._fields_:
            lines.append(f'  printf("off {st}.{name} %zu\\n", offsetof({st}, {name}));')
    for c in consts:
        lines.append(f'  printf("const {c} %d\\n", (int)({c}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    got = dict(line.rsplit(" ", 1) for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                               check=True).stdout.splitlines())
    for st, cls in fields.items():
        assert int(got[f"size {st}"]) == ctypes.sizeof(cls), st
        for name, _ in cls._fields_:
            assert int(got[f"off {st}.{name}"]) == getattr(cls, name).offset, (st, name)
    for c, v in consts.items():
        assert int(got[f"const {c}"]) == v, c


@pytest.mark.parametrize("act", [0, 1, 2, 3, 4, 16, 17, 18, 19, 20])
def test_every_activation_is_accepted_forward(act):
    st, s = G.glu_quant_fwd_sizes(fwd_args(act=act))
    assert st == G.GLU_OK and s == (64 * 256, 64 * 8, 0, 0)


@pytest.mark.parametrize("act,status", [(0, G.GLU_OK), (1, G.GLU_OK), (2, G.GLU_OK), (3, G.GLU_OK),
                                        (4, G.GLU_OK), (18, G.GLU_EINVAL), (20, G.GLU_EINVAL),
                                        (5, G.GLU_EINVAL)])
def test_backward_activations(act, status):
    # the bf16 steps are a forward-only flag for every activation
    st, _ = G.glu_quant_bwd_sizes(bwd_args(act=act))
    assert st == status


def gemm_args(**kw):
    d = dict(act=1, fmt=1, layout=1, reserved=0, M=968, H=16384, K=2048, ld_x=2048, ld_w=2048,
             x=256, w=256, q=256, s=256)
    d.update(kw)
    return G.GluQuantGemmArgs(*(d[n] for n, _ in G.GluQuantGemmArgs._fields_))


def test_gemm_sizes():
    # NVFP4: codes [M, H/2], 128x4 scales of [M, H/16] padded to 1024 rows
    st, s = G.glu_quant_gemm_sizes(gemm_args())
    assert st == 0 and s == (968 * 8192, 1024 * 1024)
    st, s = G.glu_quant_gemm_sizes(gemm_args(fmt=0))
    assert st == 0 and s == (968 * 16384, 968 * 512)
    st, s = G.glu_quant_gemm_sizes(gemm_args(fmt=4))
    assert st == 0 and s == (968 * 16384, 1024 * 512)


@pytest.mark.parametrize("kw,status", [
    (dict(K=2000, ld_x=2000, ld_w=2000), -2), (dict(H=96), -2), (dict(ld_x=1024), -2),
    (dict(fmt=2), -1), (dict(fmt=3), -1), (dict(act=17), -1), (dict(act=5), -1), (dict(layout=2), -1),
    (dict(reserved=1), -1), (dict(M=0), -1), (dict(ld_x=2052), -3), (dict(x=264), -3),
    (dict(q=0), -1)])
def test_gemm_rejections(kw, status):
    a = gemm_args(**kw)
    assert G.glu_quant_gemm_fwd(a, None) == status
    if "x" not in kw and "q" not in kw:
        assert G.glu_quant_gemm_sizes(a)[0] == status


def test_coordinate_limit_applies_to_the_quantised_formats_only():
    # BF16 / FP32 address memory with 64-bit offsets: 2^31 rows are accepted
    st, s = G.glu_quant_fwd_sizes(fwd_args(fmt=2, q_row=None, s_row=None, out=P, M=1 << 31, N=32, ld_in=32))
    assert st == G.GLU_OK and s[0] == (1 << 31) * 32 * 2
    # the largest quantised shapes inside the limit are accepted
    st, _ = G.glu_quant_fwd_sizes(fwd_args(M=(1 << 31) - 32, N=32, ld_in=32))
    assert st == G.GLU_OK
    st, _ = G.glu_quant_bwd_sizes(bwd_args(M=32, N=(1 << 30) - 32, ld_in=(1 << 30) - 32, ld_dy=(1 << 30) - 32))
    assert st == G.GLU_OK
    st, _ = G.glu_quant_bwd_sizes(bwd_args(M=32, N=1 << 30, ld_in=1 << 30, ld_dy=1 << 30))
    assert st == G.GLU_ESHAPE
