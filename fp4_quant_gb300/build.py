"""Build libglu_quant.so in-tree for sm_103a.

Steps: compile and run the activation-table generator (gcc), compile each
CUDA translation unit with nvcc in parallel (one -gencode, no fast-math, no
FMA contraction outside explicit fma calls), link a shared library with the
CUDA runtime linked statically.  Re-running is incremental (mtime based).

Usage: python -m fp4_quant_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
GEN = os.path.join(PKG, "_gen")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libglu_quant.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden"]
UNITS = ["api.cu", "tmap.cu", "fwd_mx.cu", "fwd_mx_b16.cu", "fwd_mx_x.cu", "fwd_mx_erf.cu", "bwd_mx.cu", "bwd_both.cu", "gemm_glu.cu", "plain.cu"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libglu_quant.so")


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(GEN, exist_ok=True)
    os.makedirs(BUILD, exist_ok=True)
    # 1. activation tables
    gen_src = os.path.join(CSRC, "gen_act_tables.c")
    gen_bin = os.path.join(BUILD, "gen_act_tables")
    tables = os.path.join(GEN, "act_tables.inc")
    if force or _newer(gen_bin, [gen_src]):
        _run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", gen_src, "-lm",
              "-o", gen_bin], verbose)
    if force or _newer(tables, [gen_bin]):
        out = subprocess.run([gen_bin], capture_output=True, text=True, check=True).stdout
        tmp = tables + f".tmp{os.getpid()}"
        with open(tmp, "w") as f:
            f.write(out)
        os.replace(tmp, tables)
    # 2. translation units
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, h) for h in ("glu_common.cuh", "kernels.h", "tma.cuh", "mx_block.cuh", "nv_block.cuh", "ring.cuh", "bwd_common.cuh", "fwd_mx.cuh", "tc.cuh")]
    headers += [tables, os.path.join(INCLUDE, "glu_quant.h")]
    objs, jobs = [], []
    for u in UNITS:
        src = os.path.join(CSRC, u)
        obj = os.path.join(BUILD, u.replace(".cu", ".o"))
        objs.append(obj)
        if force or _newer(obj, [src] + headers):
            jobs.append([nvcc, *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-c", src, "-o", obj])
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for f in [ex.submit(_run, j, verbose) for j in jobs]:
                f.result()
    # 3. link
    if force or jobs or _newer(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        _run([nvcc, *ARCH, "-shared", "-cudart", "static", *objs, "-o", tmp], verbose)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="--verbose" in sys.argv)
    print(LIB)
