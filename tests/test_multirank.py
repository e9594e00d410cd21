"""Multi-rank host logic of the bench on CPU (gloo, world size 2).

The path shards by rows with no exchange step: each rank processes its own
batch and the only cross-rank traffic is the barrier and the max-over-ranks
of the timed region.  This checks that aggregation with real process groups.
"""
import os
import socket

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
