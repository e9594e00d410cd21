"""Multi-rank host logic on CPU (gloo, world size 2).

The path shards by rows with no exchange step: each rank processes its own
rows and the only cross-rank traffic is the barrier and the max-over-ranks
of the timed region.  These tests check that aggregation with real process
groups, and that row slices quantised on separate ranks (by the oracle)
join to the full batch's output.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [12.5, 20.0][rank]            # rank 1 is the slow one
        dist.barrier()
        worst = bench.reduce_max(ms, dist, torch.device("cpu"))
        per_rank_bytes = 1_000_000_000
        v = bench.whole_job_gbps(world, per_rank_bytes, 4, worst)
        q.put((rank, worst, v))
    finally:
        dist.destroy_process_group()


def test_two_rank_weak_scaling_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, worst, v in res:
        assert worst == 20.0                  # every rank sees the slowest time
        assert v == pytest.approx(2 * 1e9 * 4 / 20e-3 / 1e9)


def _bf16_bits(rng, shape, spikes=0.0):
    x = rng.standard_normal(shape).astype(np.float32)
    if spikes:
        m = rng.random(shape) < spikes
        x[m] = np.where(rng.random(int(m.sum())) < 0.5, -60.0, 60.0)
    b = x.view(np.uint32)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)  # round to nearest even


def _slice_worker(rank, world, port, q):
    """Each rank runs the oracle on its own 32-row-aligned slice of one
    seeded batch (no exchange on the data path) and sends its outputs to
    rank 0, which joins them."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle as O
        rng = np.random.default_rng(77)
        M, N = 160, 96  # five 32-row blocks: ranks get 96 and 64 rows
        g, u, d = (_bf16_bits(rng, (M, N), 0.01) for _ in range(3))
        per = -(-(M // 32) // world) * 32
        r0, r1 = min(M, rank * per), min(M, (rank + 1) * per)
        mine = {
            "fwd": O.glu_fwd(g[r0:r1], u[r0:r1], act=O.SILU, fmt=O.MXFP8, mode=O.BOTH, nthreads=1),
            "bwd": O.glu_bwd(g[r0:r1], u[r0:r1], d[r0:r1], act=O.GELU_TANH, fmt=O.MXFP8, mode=O.BOTH,
                             nthreads=1),
        }
        parts = [None] * world if rank == 0 else None
        dist.gather_object((r0, r1, mine), parts, dst=0)
        if rank == 0:
            q.put(parts)
    finally:
        dist.destroy_process_group()


def test_two_rank_row_slices_join_to_the_full_batch():
    """Two gloo ranks each quantise their 32-row-aligned slice (forward and
    backward, both directions); joined (rowwise outputs by rows, colwise
    outputs [W, M] by columns) they equal the oracle's full-batch output
    byte for byte: the path shards by rows with no exchange step."""
    import oracle as O
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_slice_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    parts = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    rng = np.random.default_rng(77)
    M, N = 160, 96
    g, u, d = (_bf16_bits(rng, (M, N), 0.01) for _ in range(3))
    full = {
        "fwd": O.glu_fwd(g, u, act=O.SILU, fmt=O.MXFP8, mode=O.BOTH, nthreads=1),
        "bwd": O.glu_bwd(g, u, d, act=O.GELU_TANH, fmt=O.MXFP8, mode=O.BOTH, nthreads=1),
    }
    assert [p[:2] for p in parts] == [(0, 96), (96, 160)]
    for k in ("fwd", "bwd"):
        for key, axis in (("q_row", 0), ("s_row", 0), ("q_col", 1), ("s_col", 1)):
            joined = np.concatenate([p[2][k][key] for p in parts], axis=axis)
            assert np.array_equal(joined, full[k][key]), (k, key)


def test_single_rank_reduce_is_identity():
    assert bench.reduce_max(3.5, None, None) == 3.5
    assert bench.whole_job_gbps(1, 5_000_000_000, 2, 1000.0) == pytest.approx(10.0)


def test_algorithmic_byte_model_matches_the_page_figures():
    # the byte model reproduces the pages' GB/s from their times
    # (131072 x 8192: fwd row 904.19 us -> 5974.7 GB/s; bwd both 1859.09 us -> 5847.8 GB/s)
    M, N = 131072, 8192
    assert bench.algo_bytes("fwd", 1, M, N) / 904.19e-6 / 1e9 == pytest.approx(5974.7, abs=0.1)
    assert bench.algo_bytes("bwd", 3, M, N) / 1859.09e-6 / 1e9 == pytest.approx(5847.8, abs=0.1)
    assert bench.algo_bytes("fwd", 3, 16384, 7168) / 143.36e-6 / 1e9 == pytest.approx(4966.4, abs=0.1)


def test_algorithmic_bytes_per_format():
    # per output element: forward reads 4 B and writes 1 + 1/32 B per MXFP8
    # direction, 1/2 + 1/16 B NVFP4, 2 B bf16; backward reads 6 B and writes
    # twice that per (gate, up) element
    assert bench.algo_bytes("fwd", 1, 128, 128) == 65536 + 16896
    M, N = 131072, 8192
    assert bench.algo_bytes("fwd", 2, M, N) == bench.algo_bytes("fwd", 1, M, N) == 5402263552
    assert bench.algo_bytes("fwd", 3, M, N) == 4 * M * N + 2 * (M * N + M * N // 32)
    assert bench.algo_bytes("bwd", 1, M, N) == 6 * M * N + 2 * (M * N + M * N // 32)
    # NVFP4, interleaved GeGLU 784 x 16384 outputs: 51.38 MB read, 7.225 MB written
    assert bench.algo_bytes("fwd", 1, 784, 16384, "nvfp4") == 51380224 + 7225344
    assert bench.algo_bytes("bwd", 1, 8192, 14336, "nvfp4") == 6 * 8192 * 14336 + 8192 * 14336 * 9 // 8
    assert bench.algo_bytes("fwd", 1, 8192, 11008, "bf16") == 6 * 8192 * 11008


def test_kernel_source_hash_follows_each_kernel_own_sources():
    # every call maps to a translation unit whose includes resolve; the
    # forward and the two backward kernels are keyed separately
    hs = {tu: bench.kernel_src_hash(tu) for tu in set(bench.KERNEL_TU.values())}
    assert len(set(hs.values())) == len(hs)
    assert all(len(h) == 16 for h in hs.values())
    for d, m in (("fwd", "row"), ("bwd", "both")):
        t = bench.profiled_traffic(d, m, 131072, 8192)
        assert t is None or t > bench.algo_bytes(d, 1 if m == "row" else 3, 131072, 8192) * 0.9


def test_padded_bytes_count_the_128x4_padding():
    # C4 at 784 rows: 784 -> 896 padded rows of 1024 scale bytes
    assert bench.padded_bytes("fwd", 1, 784, 16384, "nvfp4") == 51380224 + 784 * 8192 + 896 * 1024
    # backward: [dGate | dUp] is 2N wide; 8192 rows need no row padding
    assert bench.padded_bytes("bwd", 1, 8192, 14336, "nvfp4") == bench.algo_bytes("bwd", 1, 8192, 14336, "nvfp4")
    # 40 rows, width 48: 3 scale columns padded to 4, 40 rows to 128
    assert bench.padded_bytes("fwd", 1, 40, 48, "nvfp4") == 4 * 40 * 48 + 40 * 24 + 128 * 4
    assert bench.padded_bytes("fwd", 3, 128, 128) == bench.algo_bytes("fwd", 3, 128, 128)


def test_code_hash_ignores_comments_only():
    a = 'int f(int x) {  // doubles\n  return 2 * x; /* twice */\n}\nconst char* s = "/* kept */";\n'
    b = '/* header */\nint f(int x) {\n  return 2 * x;\n}\n\nconst char* s = "/* kept */";  // note\n'
    assert bench.c_code_only(a) == bench.c_code_only(b)
    assert bench.c_code_only(a) != bench.c_code_only(a.replace("2 * x", "3 * x"))
    assert bench.c_code_only(a) != bench.c_code_only(a.replace("/* kept */", "kept"))


def test_clock_summary_reads_the_sampled_csv(tmp_path):
    # rows as nvidia-smi --format=csv,noheader,nounits writes them; the idle
    # sample (power <= 200 W) is left out of the median and the reasons
    c = bench.Clocks(0, enabled=False)
    c.path = str(tmp_path / "clocks.csv")
    c.proc = object()  # a sampler that ran
    with open(c.path, "w") as f:
        f.write("0, 1200, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 2070, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 2055, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("garbage line\n")
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
