"""Benchmark of the fused gated-GLU + block-scaled quantisation path on GB300.

Headline workload (one "step"): SwiGLU at M=131072, N=8192 (gate, up, dY
bf16 N(0,1) with 0.1% of elements set to +-60), MXFP8 E4M3/E8M0 outputs, the
six calls forward {row, col, both} and backward {row, col, both}, each its
own kernel launch.  The metric is effective bandwidth: algorithmic bytes
read + written (4 B/elem read forward, 6 B/elem backward; 1 + 1/32 B written
per element and direction) divided by device time, reported against the
measured HBM copy bandwidth.  Inputs (6 GB) are far larger than L2, so
nothing is flushed between steps.

Beside the headline line's timed steps (CUDA events around each call):
  * ``modes``: every call also timed as a CUDA graph of 20 calls per replay
    (25 warm-up replays, median and min of 30);
  * ``configs``: the other workloads (SwiGLU 128x128; SwiGLU 4096x7168 all
    six calls; GeGLU 8192 x {11008, 14336, 18944, 29568} MXFP8 rowwise and
    BF16 forward and backward; GeGLU NVFP4 interleaved at 784 and 968 rows),
    graph-timed the same way, with a cold-L2 figure (a graph rotating
    through buffer sets totalling more than twice L2) for the L2-resident
    ones;
  * ``parity``: every output of every call above compared with the CPU
    oracle on the same input bytes (the headline workload on all 131072
    rows): scale mismatches and out-of-window code mismatches must be 0,
    code mismatches inside the 2-ulp window are counted;
  * ``cpu_baseline``: the oracle's own time for the headline step on all
    host cores (and on one core, on a sample).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--no-e2e] [--no-cpu] [--no-configs] [--sweep FILE]

One JSON line on stdout (rank 0).  ``--impl reference`` times the CPU oracle
(the only reference implementation that exists for this path) on a bounded
sample of the same workload.  ``--sweep FILE`` also writes one JSONL record
per extra format and activation (128x4 scales, ReLU, identity, GELU-erf,
bf16 steps, NVFP4 backward and global scale).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused GLU+quant effective GB/s and % of GB300 HBM peak; µs/call"
M_FULL, N_FULL = 131072, 8192
CALLS = [("fwd", 1), ("fwd", 2), ("fwd", 3), ("bwd", 1), ("bwd", 2), ("bwd", 3)]
MODE_NAME = {1: "row", 2: "col", 3: "both"}
# the pages' GB200 per-call times for these six calls at 131072x8192 (context)
PAGE_GB200_US = {("fwd", 1): 904.19, ("fwd", 2): 1022.98, ("fwd", 3): 1216.08,
                 ("bwd", 1): 1321.98, ("bwd", 2): 1710.08, ("bwd", 3): 1859.09}
L2_BYTES = 129 * 2 ** 20
GRAPH_REPS, GRAPH_WARM, GRAPH_SAMPLES = 20, 25, 30


def algo_bytes(direction: str, mode: int, M: int, N: int, fmt: str = "mxfp8") -> int:
    """Algorithmic bytes of one call (read + written, unpadded)."""
    MN = M * N
    dirs = 2 if mode == 3 else 1
    if direction == "fwd":
        read = 4 * MN
        if fmt == "mxfp8":
            write = dirs * (MN + MN // 32)
        elif fmt == "nvfp4":
            write = MN // 2 + MN // 16
        elif fmt == "bf16":
            write = 2 * MN
        else:
            write = 4 * MN
    else:
        read = 6 * MN
        if fmt == "mxfp8":
            write = dirs * 2 * (MN + MN // 32)
        elif fmt == "nvfp4":
            write = MN + MN // 8
        elif fmt == "bf16":
            write = 4 * MN
        else:
            write = 8 * MN
    return read + write


def padded_bytes(direction: str, mode: int, M: int, N: int, fmt: str = "mxfp8") -> int:
    """Bytes of one call with NVFP4's scale matrix counted at its padded
    128x4 size (rows to a multiple of 128, scale columns to a multiple of
    4, the padding written as zeros); the same as algo_bytes otherwise."""
    if fmt != "nvfp4":
        return algo_bytes(direction, mode, M, N, fmt)
    W = N if direction == "fwd" else 2 * N
    scales = M * W // 16
    padded = -(-M // 128) * 128 * (-(-(W // 16) // 4) * 4)
    return algo_bytes(direction, mode, M, N, fmt) - scales + padded


def reduce_max(x: float, dist, device) -> float:
    """Max of a per-rank scalar over all ranks (identity without a group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(world: int, bytes_per_rank_step: int, steps: int, max_ms: float) -> float:
    """Weak scaling: every rank processes its own batch; the job's bandwidth
    is all ranks' bytes over the slowest rank's time."""
    return world * bytes_per_rank_step * steps / (max_ms * 1e-3) / 1e9


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "of measured (MEASURED_PEAKS.json hbm_gbs)"}
    return {"hbm_gbs": 6800.0, "source": "of fallback (6.8 TB/s)"}


# Translation unit that holds each call's kernel.
KERNEL_TU = {"fwd": "fwd_mx.cu", "bwd_row": "bwd_mx.cu", "bwd_col": "bwd_mx.cu",
             "bwd_both": "bwd_both.cu"}
# Files besides its translation unit that shape every launch: the tensor
# maps, the launch declarations and the generator of the activation tables.
# The entry points' argument checks (api.cu) are left out: they decide which
# calls run, not how a launch reads or writes memory.
KERNEL_HOST = ("tmap.cu", "kernels.h", "gen_act_tables.c")


def c_code_only(text: str) -> str:
    """C/C++ source without its comments and with whitespace runs collapsed,
    so that an edit of comments or layout leaves the hash of the code alone
    (string and character literals are kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(" ".join(line.split()) for line in "".join(out).splitlines() if line.strip())


def kernel_src_hash(tu: str) -> str:
    """Hash of the code one kernel is built from: its translation unit
    (kernel and launcher), the library headers it includes (transitively)
    and KERNEL_HOST, comments left out."""
    d = os.path.join(ROOT, "fp4_quant_gb300", "csrc")
    seen, todo = set(KERNEL_HOST), [tu]
    while todo:
        n = todo.pop()
        if n in seen:
            continue
        seen.add(n)
        with open(os.path.join(d, n)) as f:
            for line in f:
                m = re.match(r'\s*#include\s+"([^"/]+)"', line)
                if m:
                    todo.append(m.group(1))
    h = hashlib.sha256()
    for n in sorted(seen):
        with open(os.path.join(d, n)) as f:
            h.update(n.encode() + c_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(direction: str, mode: str, M: int, N: int):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the sources the kernel is built from now (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    key = f"{direction}_mx_{mode}_{M}x{N}"
    tu = KERNEL_TU.get(direction if direction == "fwd" else f"{direction}_{mode}")
    if tu is None:
        return None
    cur = kernel_src_hash(tu)
    for line in open(p):
        parts = line.split()
        if len(parts) >= 3 and parts[0] == key and parts[2] == cur:
            return float(parts[1])
    return None


class Clocks:
    """nvidia-smi sampling during the timed region."""

    def __init__(self, index: int, enabled: bool = True):
        self.proc = None
        self.enabled = enabled
        self.index = index
        self.path = os.path.join(tempfile.gettempdir(), f"glu_quant_clocks_{os.getpid()}.csv")

    def __enter__(self):
        if not self.enabled:
            return self
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                rows.append((float(p[1]), float(p[2]), float(p[3]), p[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        load = [r for r in rows if r[2] > 200.0] or rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in load:
            for n, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in load),
                "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(load)}


# ------------------------------------------------------------ GPU timing --

def graph_time(fns, dev, reps=GRAPH_REPS, warm=GRAPH_WARM, samples=GRAPH_SAMPLES):
    """Median and min µs per call of a CUDA graph that runs the calls
    ``fns`` (each takes a stream handle) in turn until it holds ``reps``
    calls (a list longer than ``reps`` is captured whole)."""
    import torch
    n = max(reps, len(fns))
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for f in fns:  # eager warm-up on the capture stream (lazy set-up)
            f(s.cuda_stream)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for i in range(n):
                fns[i % len(fns)](s.cuda_stream)
    torch.cuda.synchronize(dev)
    for _ in range(warm):
        graph.replay()
    torch.cuda.synchronize(dev)
    out = []
    for _ in range(samples):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        b.synchronize()
        out.append(a.elapsed_time(b) * 1e3 / n)
    del graph
    return statistics.median(out), min(out)


def device_error_bits(G) -> dict:
    """Error bits the kernels' bounded waits recorded (then cleared): a wait
    that gave up leaves partial output behind, so any bit voids the timing."""
    st, f, b = G.glu_quant_device_errors(clear=True)
    return {"status": st, "fwd": f, "bwd": b, "ok": st == 0 and f == 0 and b == 0}


# ----------------------------------------------------------- parity (host) --

def _parity_util():
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import parity_util
    return parity_util


def oracle_call(O, direction, mode, fmt, act, bits, layout=0, N=None, nthreads=None):
    """The oracle's outputs of one call on host bit arrays (gate, up, dy)."""
    gb, ub, db = bits
    ofmt = {"mxfp8": O.MXFP8, "nvfp4": O.NVFP4, "bf16": O.BF16, "fp32": O.FP32}[fmt]
    if direction == "fwd":
        return O.glu_fwd(gb, ub, act=act, fmt=ofmt, mode=mode, layout=layout, N=N, nthreads=nthreads)
    return O.glu_bwd(gb, ub, db, act=act, fmt=ofmt, mode=mode, layout=layout, N=N, nthreads=nthreads)


def parity_of(O, PU, direction, mode, fmt, act, bits, gpu_host, M, N, layout=0, ref=None):
    """Counts of one call's comparison with the oracle (PU.compare_counts)."""
    ofmt = {"mxfp8": O.MXFP8, "nvfp4": O.NVFP4, "bf16": O.BF16}[fmt]
    if ref is None:
        ref = oracle_call(O, direction, mode, fmt, act, bits, layout, N)
    W = N if direction == "fwd" else 2 * N

    def h_rows(rows):
        gb, ub, db = bits
        sub = lambda x: None if x is None else x[rows]
        return oracle_call(O, direction, 1, "fp32", act, (sub(gb), sub(ub), sub(db)), layout, N)["out"]
    return PU.compare_counts(gpu_host, ref, ofmt, mode, M, W, h_rows)


def host_outputs(o: dict) -> dict:
    """Host numpy copies of a call's output tensors."""
    import torch
    r = {}
    for k, t in o.items():
        if t is None:
            r[k] = None
        elif t.dtype == torch.bfloat16:
            r[k] = t.contiguous().view(torch.int16).cpu().numpy().view("uint16")
        else:
            r[k] = t.cpu().numpy()
    return r


# ------------------------------------------------------------------ GPU arm --

def gpu_arm(args, rank, world, dist):
    import torch

    import fp4_quant_gb300 as G
    import synth

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    sp = synth.spec("swiglu_131072", M=args.rows)
    M, N = sp.M, sp.N
    calls = [c for c in CALLS if f"{c[0]}_{MODE_NAME[c[1]]}" in args.calls.split(",")] \
        if args.calls else CALLS
    x = synth.make(sp, dev, with_dy=True, seed_offset=rank * 10)
    g, u, d = x["gate"], x["up"], x["dy"]

    # preallocated outputs for each of the six calls
    def outs(direction, mode):
        W = N if direction == "fwd" else 2 * N
        o = {"q_row": None, "s_row": None, "q_col": None, "s_col": None, "out": None}
        if mode & 1:
            o["q_row"] = torch.empty((M, W), dtype=torch.uint8, device=dev)
            o["s_row"] = torch.empty((M, W // 32), dtype=torch.uint8, device=dev)
        if mode & 2:
            o["q_col"] = torch.empty((W, M), dtype=torch.uint8, device=dev)
            o["s_col"] = torch.empty((W, M // 32), dtype=torch.uint8, device=dev)
        return o

    bufs = {c: outs(*c) for c in calls}
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def call(c, s=None):
        direction, mode = c
        s = sh if s is None else s
        if direction == "fwd":
            G.fwd(g, u, act=G.ACT_SILU, fmt=G.FMT_MXFP8, mode=mode, out=bufs[c], stream=s)
        else:
            G.bwd(g, u, d, act=G.ACT_SILU, fmt=G.FMT_MXFP8, mode=mode, out=bufs[c], stream=s)

    def barrier():
        if dist is not None:
            dist.barrier()

    G.glu_quant_device_errors(clear=True)
    for _ in range(args.warmup):
        for c in calls:
            call(c)
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in calls] for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    with Clocks(dev.index, enabled=not args.no_clocks) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        t0.record(stream)
        for k in range(K):
            for i, c in enumerate(calls):
                ev[k][i][0].record(stream)
                call(c)
                ev[k][i][1].record(stream)
                launches += 1
        t1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    errs = device_error_bits(G)
    total_ms = t0.elapsed_time(t1)
    per_call_ms = {c: [ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(K)]
                   for i, c in enumerate(calls)}
    total_ms = reduce_max(total_ms, dist, dev)

    step_bytes = sum(algo_bytes(dr, m, M, N) for dr, m in calls)
    value = whole_job_gbps(world, step_bytes, K, total_ms)
    peaks = measured_peaks()
    modes = {}
    for c in calls:
        avg = statistics.mean(per_call_ms[c])
        gbps = algo_bytes(c[0], c[1], M, N) / (avg * 1e-3) / 1e9
        modes[f"{c[0]}_{MODE_NAME[c[1]]}"] = {
            "us": round(avg * 1e3, 2), "us_min": round(min(per_call_ms[c]) * 1e3, 2),
            "gbps": round(gbps, 1), "frac_hbm": round(gbps / peaks["hbm_gbs"], 4),
            "page_gb200_us": PAGE_GB200_US[c]}
    dom = max(calls, key=lambda c: statistics.mean(per_call_ms[c]))
    dom_name = f"{dom[0]}_{MODE_NAME[dom[1]]}"
    dom_gbps = modes[dom_name]["gbps"]
    traffic = profiled_traffic(dom[0], MODE_NAME[dom[1]], M, N)

    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(total_ms / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": bench_config(M, N, calls, world),
        "modes": modes,
        "roofline": {"bound": "hbm", "achieved": dom_gbps, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(dom_gbps / peaks["hbm_gbs"], 4),
                     "traffic": traffic, "kernel": dom_name,
                     "algo_bytes_per_launch": algo_bytes(dom[0], dom[1], M, N),
                     "peak_source": peaks["source"]},
        "page_context": {"gb200_same_calls_gbps": round(
            sum(algo_bytes(dr, m, M_FULL, N_FULL) for dr, m in CALLS)
            / (sum(PAGE_GB200_US.values()) * 1e-6) / 1e9, 1),
            "note": "the pages' GB200 per-call times for the same six calls (context, not a target)"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "device_errors": errs,
    }

    # every call also as a CUDA graph of 20 calls per replay
    if not args.no_graph:
        for c in calls:
            med, mn = graph_time([lambda s, c=c: call(c, s)], dev)
            r = modes[f"{c[0]}_{MODE_NAME[c[1]]}"]
            r["us_graph"] = round(med, 2)
            r["us_graph_min"] = round(mn, 2)
            r["frac_hbm_graph"] = round(algo_bytes(c[0], c[1], M, N) / (med * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)
        res["device_errors_graph"] = device_error_bits(G)

    host_in = gpu_out = None
    if rank == 0 and (not args.no_parity or (not args.no_cpu and world == 1)):
        host_in = [synth.to_host_bits(t) for t in (g, u, d)]
        if not args.no_parity:
            gpu_out = {c: host_outputs(bufs[c]) for c in calls}

    if not args.no_e2e:
        res["e2e"] = e2e_leg(args, G, g, u, d, bufs, calls, dev, stream, dist, world, step_bytes)
    del x, g, u, d, bufs
    torch.cuda.empty_cache()

    if not args.no_configs and rank == 0:
        res["configs"] = configs_block(args, G, dev, peaks, parity=not args.no_parity)
        res["gemm"] = gemm_block(G, dev, parity=not args.no_parity)
        res["device_errors_configs"] = device_error_bits(G)
    return res, host_in, gpu_out, (M, N, calls)


def e2e_leg(args, G, g, u, d, bufs, calls, dev, stream, dist, world, step_bytes):
    """The same six calls through the public API with host buffers: every
    step copies the inputs host->device from pinned memory and reads every
    call's outputs back, inside the timed region."""
    import torch
    hg = torch.empty(g.shape, dtype=g.dtype, pin_memory=True)
    hu = torch.empty(u.shape, dtype=u.dtype, pin_memory=True)
    hd = torch.empty(d.shape, dtype=d.dtype, pin_memory=True)
    hg.copy_(g)
    hu.copy_(u)
    hd.copy_(d)
    biggest = max(calls, key=lambda c: sum(t.numel() for t in bufs[c].values() if t is not None))
    hout = {k: (torch.empty(t.shape, dtype=t.dtype, pin_memory=True) if t is not None else None)
            for k, t in bufs[biggest].items()}
    h2d = sum(t.numel() * t.element_size() for t in (hg, hu, hd))
    d2h = sum(sum(t.numel() * t.element_size() for t in bufs[c].values() if t is not None)
              for c in calls)
    sh = stream.cuda_stream

    def step():
        g.copy_(hg, non_blocking=True)
        u.copy_(hu, non_blocking=True)
        d.copy_(hd, non_blocking=True)
        for c in calls:
            direction, mode = c
            if direction == "fwd":
                G.fwd(g, u, act=G.ACT_SILU, fmt=G.FMT_MXFP8, mode=mode, out=bufs[c], stream=sh)
            else:
                G.bwd(g, u, d, act=G.ACT_SILU, fmt=G.FMT_MXFP8, mode=mode, out=bufs[c], stream=sh)
            for k, t in bufs[c].items():
                if t is not None:
                    hout[k].view(-1)[: t.numel()].copy_(t.view(-1), non_blocking=True)

    step()
    torch.cuda.synchronize(dev)
    K = max(1, min(args.steps, 3))
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0.record(stream)
    for _ in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    ms = reduce_max(t0.elapsed_time(t1), dist, dev)
    return {"value": round(whole_job_gbps(world, step_bytes, K, ms), 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "ms_per_step": round(ms / K, 3)}


# ------------------------------------------------------ the other configs --

def config_calls(G):
    """(config, workload spec args, [(direction, mode, fmt, act, layout)]),
    the shapes and calls of the non-headline workloads."""
    S, GE = G.ACT_SILU, G.ACT_GELU_TANH
    c3 = [("fwd", 1, "mxfp8", GE, 0), ("bwd", 1, "mxfp8", GE, 0),
          ("fwd", 1, "bf16", GE, 0), ("bwd", 1, "bf16", GE, 0)]
    return ([("C1", ("swiglu_128", {}), [("fwd", 1, "mxfp8", S, 0)])]
            + [("C2", ("swiglu_4096", {}), [(dr, m, "mxfp8", S, 0) for dr in ("fwd", "bwd") for m in (1, 2, 3)])]
            + [("C3", ("geglu_8192", {"N": n}), c3) for n in (11008, 14336, 18944, 29568)]
            + [("C4", ("geglu_nvfp4", {"M": m}), [("fwd", 1, "nvfp4", GE, 1)]) for m in (784, 968)])


def configs_block(args, G, dev, peaks, parity=True):
    """Graph-timed µs, GB/s and fraction of HBM per call of every config,
    cold-L2 figures where the working set fits in L2, parity counts."""
    import torch

    import oracle as O
    import synth
    PU = _parity_util() if parity else None
    fmts = {"mxfp8": G.FMT_MXFP8, "nvfp4": G.FMT_NVFP4, "bf16": G.FMT_BF16}
    oact = {G.ACT_SILU: O.SILU, G.ACT_GELU_TANH: O.GELU_TANH}
    recs = []
    for cname, (wl, kw), cl in config_calls(G):
        sp = synth.spec(wl, **kw)
        x = synth.make(sp, dev, with_dy=any(dr == "bwd" for dr, *_ in cl))
        interleaved = sp.interleaved
        gin, uin = (x["x"], None) if interleaved else (x["gate"], x["up"])
        din = x.get("dy")
        M, N = sp.M, sp.N
        bits = None
        if parity:
            tb = lambda t: None if t is None else synth.to_host_bits(t)
            bits = (tb(gin), tb(uin), tb(din))
        for (dr, mode, fmt, act, layout) in cl:
            f = fmts[fmt]
            mk = lambda s, o=None, dr=dr, mode=mode, f=f, act=act, layout=layout, gin=gin, uin=uin, din=din: (
                G.fwd(gin, uin, act=act, fmt=f, mode=mode, layout=layout, out=o, stream=s) if dr == "fwd"
                else G.bwd(gin, uin, din, act=act, fmt=f, mode=mode, layout=layout, out=o, stream=s))
            o = mk(None)
            med, mn = graph_time([lambda s, o=o, mk=mk: mk(s, o)], dev)
            nbytes = algo_bytes(dr, mode, M, N, fmt)
            gbps = nbytes / (med * 1e-6) / 1e9
            r = {"config": cname, "workload": wl, "direction": dr, "mode": MODE_NAME[mode], "fmt": fmt,
                 "act": "silu" if act == G.ACT_SILU else "gelu_tanh",
                 "layout": "interleaved" if layout else "split", "M": M, "N": N,
                 "us_graph": round(med, 3), "us_graph_min": round(mn, 3), "bytes": nbytes,
                 "gbps": round(gbps, 1), "frac_hbm": round(gbps / peaks["hbm_gbs"], 4),
                 "l2_resident": nbytes < L2_BYTES}
            if fmt == "nvfp4":
                pb = padded_bytes(dr, mode, M, N, fmt)
                r.update({"bytes_padded": pb, "gbps_padded": round(pb / (med * 1e-6) / 1e9, 1)})
            if nbytes < L2_BYTES:
                r.update(cold_l2(G, dev, sp, dr, mode, f, act, layout, nbytes, peaks))
            torch.cuda.synchronize(dev)
            if parity:
                gpu_host = host_outputs(o)
                r["parity"] = parity_of(O, PU, dr, mode, fmt, oact[act], bits, gpu_host, M, N, layout=layout)
            recs.append(r)
            print(json.dumps(r), file=sys.stderr, flush=True)
            del o
        del x, gin, uin, din
        torch.cuda.empty_cache()
    return recs


def cold_l2(G, dev, sp, dr, mode, f, act, layout, nbytes, peaks):
    """µs per call with every call of the graph on its own input/output set,
    at least 4 sets and more than 2x L2 in all, so that no call finds its
    data in L2."""
    import torch

    import synth
    sets = max(4, -(-2 * L2_BYTES // nbytes) + 1)
    ins = []
    base = synth.make(sp, dev, with_dy=dr == "bwd")
    for i in range(sets):
        # one copy per set (the values do not matter for the timing)
        ins.append({k: v.clone() for k, v in base.items()})
    fns = []
    for xi in ins:
        gin, uin = (xi["x"], None) if sp.interleaved else (xi["gate"], xi["up"])
        din = xi.get("dy")
        mk = lambda s, o=None, gin=gin, uin=uin, din=din: (
            G.fwd(gin, uin, act=act, fmt=f, mode=mode, layout=layout, out=o, stream=s) if dr == "fwd"
            else G.bwd(gin, uin, din, act=act, fmt=f, mode=mode, layout=layout, out=o, stream=s))
        o = mk(None)
        fns.append(lambda s, mk=mk, o=o: mk(s, o))
    med, mn = graph_time(fns, dev, reps=len(fns), warm=5, samples=15)
    del ins, fns, base
    torch.cuda.empty_cache()
    gbps = nbytes / (med * 1e-6) / 1e9
    return {"cold_l2": {"us": round(med, 3), "us_min": round(mn, 3), "gbps": round(gbps, 1),
                        "frac_hbm": round(gbps / peaks["hbm_gbs"], 4), "buffer_sets": sets,
                        "bytes_all_sets": sets * nbytes}}


# ------------------------------------------- the gate/up GEMM with the quantiser --

def measured_bf16_tflops() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"tflops": float(d["bf16_tflops"]), "source": "of measured (MEASURED_PEAKS.json bf16_tflops, burst)"}
    return {"tflops": 1900.0, "source": "of fallback (1.9 PFLOP/s bf16 burst)"}


def gemm_block(G, dev, parity=True):
    """The pages' fused GEMM shapes (pi0.5 MLP: M in {784, 968}, K = 2048,
    merged N = 32768, H = 16384), bf16 operands, GeGLU (tanh), NVFP4 output,
    interleaved gate/up rows: CUDA-graph-timed µs per call and tensor
    throughput (2 M 2H K flops) against the measured bf16 peak; parity on the
    first row tile (the tensor cores' fp32 accumulation order may move a
    value next to a rounding boundary by one step)."""
    import numpy as np
    import torch
    peak = measured_bf16_tflops()
    recs = []
    for M in (784, 968):
        H, K = 16384, 2048
        g = torch.Generator(device=dev).manual_seed(5000 + M)
        x = torch.randn(M, K, generator=g, device=dev).to(torch.bfloat16)
        w = (torch.randn(2 * H, K, generator=g, device=dev) / 32).to(torch.bfloat16)
        o = G.gemm(x, w, act=G.ACT_GELU_TANH, fmt=G.FMT_NVFP4, layout=G.LAYOUT_INTERLEAVED)
        med, mn = graph_time([lambda st, o=o: G.gemm(x, w, act=G.ACT_GELU_TANH, fmt=G.FMT_NVFP4,
                                                     layout=G.LAYOUT_INTERLEAVED, out=o, stream=st)], dev)
        flops = 2 * M * 2 * H * K
        tf = flops / (med * 1e-6) / 1e12
        r = {"workload": f"geglu_gemm_nvfp4_{M}x{H}_k{K}", "M": M, "H": H, "K": K, "act": "gelu_tanh",
             "fmt": "nvfp4", "layout": "interleaved", "operands": "bf16", "us_graph": round(med, 3),
             "us_graph_min": round(mn, 3), "flops": flops, "tflops": round(tf, 1),
             "frac_bf16_peak": round(tf / peak["tflops"], 4), "peak_source": peak["source"]}
        if parity:
            import oracle as O
            torch.cuda.synchronize(dev)
            xb = x[:128].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
            wb = w.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
            ref = O.gemm_glu_fwd(xb, wb, act=O.GELU_TANH, fmt=O.NVFP4, layout=O.INTERLEAVED)
            q = o["q"][: 128 * H // 2].cpu().numpy().reshape(128, H // 2)
            sg = o["s"][: 128 * H // 16].cpu().numpy()
            un = lambda t: np.stack([t & 0xF, t >> 4], axis=-1).reshape(t.shape[0], -1)
            cg, cr = un(q), un(ref["q"])
            diff = cg != cr
            a, b = cg[diff], cr[diff]
            one_step = (((a & 8) == (b & 8)) & (np.abs((a & 7).astype(int) - (b & 7).astype(int)) == 1)) | \
                       (((a & 7) == 0) & ((b & 7) == 0))
            r["parity_first_row_tile"] = {
                "elements": int(cg.size), "code_mismatches": int(diff.sum()),
                "more_than_one_step": int((~one_step).sum()), "scales": int(sg.size),
                "scale_mismatches": int((sg != ref["s"]).sum()),
                "rule": "tensor-core fp32 accumulation vs the oracle's correctly rounded sums: "
                        "codes may differ by one step next to a boundary"}
        recs.append(r)
        print(json.dumps(r), file=sys.stderr, flush=True)
        del x, w, o
        torch.cuda.empty_cache()
    return recs


# ------------------------------------------------------------- CPU (oracle) --

_SAMPLE_CACHE = {}


def oracle_sample(rows: int, seed_offset: int = 0, nthreads: int | None = None):
    """Time the oracle on `rows` rows of the same workload (host inputs drawn
    once with the same generator recipe, on the CPU; drawing is not timed)."""
    import oracle as O
    import synth
    key = (rows, seed_offset)
    if key not in _SAMPLE_CACHE:
        sp = synth.spec("swiglu_131072", M=rows)
        x = synth.make(sp, "cpu", with_dy=True, seed_offset=seed_offset)
        _SAMPLE_CACHE.clear()
        _SAMPLE_CACHE[key] = (sp, [synth.to_host_bits(x[k]) for k in ("gate", "up", "dy")])
    sp, (gb, ub, db) = _SAMPLE_CACHE[key]
    nthreads = nthreads or os.cpu_count() or 1
    O.lib()
    t0 = time.perf_counter()
    for direction, mode in CALLS:
        if direction == "fwd":
            O.glu_fwd(gb, ub, act=O.SILU, fmt=O.MXFP8, mode=mode, nthreads=nthreads)
        else:
            O.glu_bwd(gb, ub, db, act=O.SILU, fmt=O.MXFP8, mode=mode, nthreads=nthreads)
    dt = time.perf_counter() - t0
    nbytes = sum(algo_bytes(dr, m, rows, sp.N) for dr, m in CALLS)
    return nbytes / dt / 1e9, dt, nthreads


def cpu_leg(host_in, gpu_out, shape, parity: bool, one_thread_rows: int):
    """The oracle on the GPU run's own input bytes: the headline step on all
    host cores, timed call by call (cpu_baseline), each call's outputs
    compared with the GPU's (parity); then a one-core sample."""
    import oracle as O
    PU = _parity_util() if parity else None
    M, N, calls = shape
    n = os.cpu_count() or 1
    O.lib()
    total, par = 0.0, {}
    for c in calls:
        dr, mode = c
        t0 = time.perf_counter()
        ref = oracle_call(O, dr, mode, "mxfp8", O.SILU, host_in, nthreads=n)
        total += time.perf_counter() - t0
        if parity:
            par[f"{dr}_{MODE_NAME[mode]}"] = parity_of(O, PU, dr, mode, "mxfp8", O.SILU, host_in,
                                                       gpu_out[c], M, N, ref=ref)
        del ref
    nbytes = sum(algo_bytes(dr, m, M, N) for dr, m in calls)
    cpu = {"value": round(nbytes / total / 1e9, 3), "unit": "GB/s", "cores": n, "kind": "oracle",
           "sample": f"all {M} rows of the timed workload's own inputs, all {len(calls)} calls, "
                     f"{total:.1f} s wall"}
    # one core, on the first rows
    r1 = min(one_thread_rows, M)
    sub = tuple(x[:r1] for x in host_in)
    t0 = time.perf_counter()
    for dr, mode in calls:
        oracle_call(O, dr, mode, "mxfp8", O.SILU, sub, nthreads=1)
    dt = time.perf_counter() - t0
    cpu["one_core"] = {"value": round(sum(algo_bytes(dr, m, r1, N) for dr, m in calls) / dt / 1e9, 3),
                       "unit": "GB/s", "cores": 1, "sample": f"first {r1} rows, all {len(calls)} calls, "
                                                             f"{dt:.1f} s wall"}
    if parity:
        par["all_ok"] = all(v["ok"] for v in par.values())
        par["rule"] = ("scales bit-exact; codes bit-exact except within 2 fp32 ulps of a rounding "
                       "boundary (one code step, counted as window)")
    return cpu, (par if parity else None)


def bench_config(M, N, calls, world):
    """The workload description both arms report."""
    return {"workload": f"swiglu_{M}x{N}_mxfp8_" + "+".join(f"{c[0]}_{MODE_NAME[c[1]]}" for c in calls),
            "M": M, "N": N, "act": "silu", "fmt": "mxfp8_e4m3_e8m0_rceil",
            "calls_per_step": len(calls), "global_batch_rows": world * M,
            "parallelism": f"dp{world}" if world > 1 else "single",
            "l2": f"inputs {6 * M * N / 1e9:.2g} GB (gate, up, dY) vs 129 MB L2; no flush"}


def reference_arm(args, rank, world):
    rows = args.ref_rows
    for _ in range(max(args.warmup, 1)):
        oracle_sample(rows)  # warm-up (page in, thread start)
    vals, times = [], []
    for _ in range(args.steps):
        v, dt, n = oracle_sample(rows)
        vals.append(v)
        times.append(dt)
    value = statistics.median(vals)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(statistics.median(times) * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": dict(bench_config(M_FULL, N_FULL, CALLS, world), sample_rows=rows),
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": n,
                             "kind": "oracle",
                             "sample": f"{rows} of 131072 rows per step, all six calls"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- sweep --

def sweep(path: str):
    """Per-format and per-activation records beyond the configs (CUDA graph
    of 20 calls per replay, 25 warm-up replays, 30 samples)."""
    import torch

    import fp4_quant_gb300 as G
    import synth
    dev = torch.device("cuda", 0)
    peaks = measured_peaks()
    recs = []

    def record(workload, direction, mode, fmt, act, M, N, fn):
        med, mn = graph_time([fn], dev)
        nbytes = algo_bytes(direction, mode, M, N, fmt)
        gbps = nbytes / (med * 1e-6) / 1e9
        r = {"workload": workload, "direction": direction, "mode": MODE_NAME.get(mode, "row"),
             "fmt": fmt, "act": act, "M": M, "N": N, "us_median": round(med, 3),
             "us_min": round(mn, 3), "bytes": nbytes, "gbps": round(gbps, 1),
             "frac_hbm": round(gbps / peaks["hbm_gbs"], 4),
             "l2_resident": nbytes < L2_BYTES}
        if fmt == "nvfp4":
            pb = padded_bytes(direction, mode, M, N, fmt)
            r.update({"bytes_padded": pb, "gbps_padded": round(pb / (med * 1e-6) / 1e9, 1)})
        recs.append(r)
        print(json.dumps(r), file=sys.stderr, flush=True)

    x = synth.make(synth.spec("swiglu_131072"), dev, with_dy=True)
    M5, N5 = x["gate"].shape
    for direction, mode in (("fwd", 3), ("bwd", 1), ("bwd", 3)):
        f = lambda s, o, dr=direction, m=mode: (
            G.fwd(x["gate"], x["up"], fmt=G.FMT_MXFP8_128X4, mode=m, out=o, stream=s) if dr == "fwd" else
            G.bwd(x["gate"], x["up"], x["dy"], fmt=G.FMT_MXFP8_128X4, mode=m, out=o, stream=s))
        o = f(None, None)
        record("swiglu_131072_mxfp8_128x4", direction, mode, "mxfp8", "silu", M5, N5,
               lambda s, f=f, o=o: f(s, o))
    for act, name in ((G.ACT_RELU, "reglu_131072"), (G.ACT_IDENTITY, "bilinear_131072"),
                      (G.ACT_GELU_ERF, "geglu_erf_131072")):
        for direction, mode in (("fwd", 1), ("fwd", 3), ("bwd", 1), ("bwd", 3)):
            f = lambda s, o, dr=direction, m=mode, a=act: (
                G.fwd(x["gate"], x["up"], act=a, mode=m, out=o, stream=s) if dr == "fwd" else
                G.bwd(x["gate"], x["up"], x["dy"], act=a, mode=m, out=o, stream=s))
            o = f(None, None)
            record(name, direction, mode, "mxfp8",
                   {G.ACT_RELU: "relu", G.ACT_IDENTITY: "identity"}.get(act, "gelu_erf"), M5, N5,
                   lambda s, f=f, o=o: f(s, o))
            del o
    for mode in (1, 3):
        o = G.fwd(x["gate"], x["up"], act=G.ACT_SILU | G.ACT_BF16_STEPS, mode=mode)
        record("swiglu_131072_bf16_steps", "fwd", mode, "mxfp8", "silu", M5, N5,
               lambda s, m=mode, o=o: G.fwd(x["gate"], x["up"], act=G.ACT_SILU | G.ACT_BF16_STEPS,
                                            mode=m, out=o, stream=s))
    del x
    for N in (14336,):
        x = synth.make(synth.spec("geglu_8192", N=N), dev, with_dy=True)
        o = G.bwd(x["gate"], x["up"], x["dy"], act=1, fmt=G.FMT_NVFP4)
        record("geglu_8192_nvfp4_bwd", "bwd", 1, "nvfp4", "gelu_tanh", 8192, N,
               lambda s, o=o: G.bwd(x["gate"], x["up"], x["dy"], act=1, fmt=G.FMT_NVFP4, out=o, stream=s))
        del x
    for M in (784, 968):
        X = synth.make(synth.spec("geglu_nvfp4", M=M), dev)["x"]
        amax = torch.tensor([50.0], dtype=torch.float32, device=dev)
        o = G.fwd(X, None, act=1, fmt=G.FMT_NVFP4, layout=1, amax=amax)
        record("geglu_nvfp4_global_scale", "fwd", 1, "nvfp4", "gelu_tanh", M, 16384,
               lambda s, o=o: G.fwd(X, None, act=1, fmt=G.FMT_NVFP4, layout=1, out=o, stream=s, amax=amax))
    with open(path, "w") as f:
        for r in recs:
            f.write(json.dumps(r) + "\n")


# ----------------------------------------------------------------- main --

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the graph-timed per-call figures")
    ap.add_argument("--no-configs", action="store_true", help="skip the non-headline configs")
    ap.add_argument("--no-parity", action="store_true", help="skip the comparisons with the oracle")
    ap.add_argument("--gemm-only", action="store_true",
                    help="only the fused gate/up GEMM block (no parity): for profiling its kernel")
    ap.add_argument("--one-core-rows", type=int, default=1024)
    ap.add_argument("--ref-rows", type=int, default=2048)
    ap.add_argument("--sweep", default=None)
    ap.add_argument("--rows", type=int, default=M_FULL,
                    help="rows of the SwiGLU workload (smaller cases for profiling)")
    ap.add_argument("--calls", default="",
                    help="comma-separated subset of fwd_row,fwd_col,fwd_both,bwd_row,bwd_col,bwd_both")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        # the oracle runs on host cores; under torchrun only rank 0 works
        if rank == 0:
            print(json.dumps(reference_arm(args, rank, world)), flush=True)
        return

    if args.gemm_only:
        import torch

        import fp4_quant_gb300 as G
        print(json.dumps({"gemm": gemm_block(G, torch.device("cuda", 0), parity=False)}), flush=True)
        return

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    res, host_in, gpu_out, shape = gpu_arm(args, rank, world, dist)
    if rank == 0 and (not args.no_parity or (not args.no_cpu and world == 1)):
        cpu, par = cpu_leg(host_in, gpu_out, shape, parity=not args.no_parity,
                           one_thread_rows=args.one_core_rows)
        if not args.no_cpu and world == 1:
            res["cpu_baseline"] = cpu
        if par is not None:
            res["parity"] = par
    if args.sweep and rank == 0:
        sweep(args.sweep)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
