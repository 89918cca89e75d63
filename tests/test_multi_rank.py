"""The multi-GPU path of bench.py on the CPU: two gloo ranks.

With N GPUs every rank runs an independent replica of the GEMM (output tiles
are independent; there is no exchange step), the timed region of the
slowest rank is taken, and the job value is all ranks' flops over that time.
These tests run that host logic with world_size 2 over gloo; the reference
arm must do its work on rank 0 only.
"""
from __future__ import annotations

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        local_ms = 10.0 + 5.0 * rank                  # rank 1 is the slow one
        slowest = bench.max_over_ranks(local_ms, torch.device("cpu"))
        value = bench.job_value(world, 2.0 * 8192 ** 3, 100, slowest)
        # the reference arm: rank 0 alone works and prints
        buf = io.StringIO()
        with redirect_stdout(buf):
            if rank != 0:
                bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1",
                                                      "--warmup", "0"]))
        q.put((rank, slowest, value, buf.getvalue()))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    expect_value = 2 * 2.0 * 8192 ** 3 * 100 / (15.0e-3) / 1e12
    for rank, slowest, value, out in results:
        assert slowest == 15.0
        assert value == pytest.approx(expect_value)
    # rank 1's reference arm printed nothing and did no work
    assert results[1][3] == ""


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, torch.device("cpu")) == 12.5
    assert bench.job_value(1, 1e12, 10, 1000.0) == pytest.approx(10.0)
