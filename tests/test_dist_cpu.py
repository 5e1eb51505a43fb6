"""The multi-GPU mode of bench.py runs one independent replica per rank (the
(batch, head) units need no exchange), so its only cross-rank step is the
timing reduction: the job lasts as long as its slowest rank and does
world_size times the work.  Checked here with two gloo ranks on the CPU."""

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 150.0][rank]
        max_ms, value = bench.job_throughput(local_ms, steps=10, units_per_step=1000, world=world, dist=dist,
                                             device="cpu")
        dist.barrier()
        q.put((rank, max_ms, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_throughput_takes_slowest_rank():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, max_ms, value in res:
        assert max_ms == 150.0
        assert value == pytest.approx(2 * 1000 * 10 / 0.150)
    del torch


def test_single_rank_without_process_group():
    pytest.importorskip("torch")
    sys.path.insert(0, ROOT)
    import bench
    max_ms, value = bench.job_throughput(50.0, steps=5, units_per_step=10, world=1, dist=None, device="cpu")
    assert max_ms == 50.0 and value == pytest.approx(5 * 10 / 0.05)
