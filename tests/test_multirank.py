"""The bench's N > 1 path on the CPU: independent replicas, one process per rank,
joined only by the max-over-ranks timing (gloo, world size 2, 127.0.0.1)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_max = bench.max_over_ranks(times[rank], "cpu", world)
        out[rank] = (ms_max, bench.whole_job_rate(1000, world, ms_max))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    import torch.multiprocessing as mp
    world, times = 2, [3.0, 5.0]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms_max, rate = res[r]
        assert ms_max == 5.0                              # every rank sees the slowest time
        assert rate == pytest.approx(2 * 1000 / 5e-3)      # units of all ranks / that time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, "cpu", 1) == 2.5
    assert bench.whole_job_rate(100, 1, 2.0) == pytest.approx(50000.0)
