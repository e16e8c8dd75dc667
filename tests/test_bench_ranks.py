"""bench.py's multi-replica aggregation on two gloo ranks (CPU): the job's step
time is the slowest rank's, and the job value counts every replica's work."""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(1.0 + rank, world, "cpu")
    out.put((rank, ms, bench.job_value(ms, world)))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import bench
    assert [r[1] for r in res] == [2.0, 2.0]
    assert res[0][2] == pytest.approx(2 * bench.CALLS * bench.product_bytes(4096, 2048) / 2e-3 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_value(1.0, 1) == pytest.approx(bench.CALLS * bench.product_bytes(4096, 2048) / 1e-3 / 1e9)
