"""The N > 1 path of bench.py on the CPU: two gloo ranks run the same
barrier / max-over-ranks reduction the timed region uses, so the reported
time is the slowest rank's and the value counts every rank's tokens."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        elapsed_ms = 10.0 + 5.0 * rank             # the second rank is the slow one
        slowest = bench.max_over_ranks(elapsed_ms, world)
        out[rank] = slowest
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_time():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1] == 15.0


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
