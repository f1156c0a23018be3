"""The multi-process path of the benchmark without a GPU: two gloo ranks on
127.0.0.1 reduce their timings the way bench.py does under torchrun (the
slowest rank's elapsed time, world x the slowest rank's end-to-end rate), and
the reference arm runs on rank 0 only."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: elapsed 1 + r seconds, end-to-end rate 100 (r + 1) queries/s
        elapsed, e2e = bench.aggregate_ranks(1.0 + rank, 100.0 * (rank + 1), world, "cpu")
        elapsed_none, e2e_none = bench.aggregate_ranks(0.5 * (rank + 1), None, world, "cpu")
        value = bench.job_throughput(64, 10, world, elapsed)
        ref = bench.run_reference(type("A", (), {"seed": 0, "workload": "tiny", "steps": 1,
                                                   "warmup": 0})(), rank, world)
        q.put((rank, elapsed, e2e, elapsed_none, e2e_none, value, ref is None))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_benchmark():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=240) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    for rank, elapsed, e2e, elapsed_none, e2e_none, value, ref_none in got:
        assert elapsed == 2.0                       # the slowest rank
        assert e2e == 200.0                         # world x the slowest rank's rate
        assert elapsed_none == 1.0 and e2e_none is None
        assert value == pytest.approx(2 * 64 * 10 / 2.0)
        assert ref_none == (rank != 0)              # the reference arm: rank 0 only


def test_single_rank_passes_through():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.aggregate_ranks(1.5, 7.0, 1, "cpu") == (1.5, 7.0)
    assert bench.job_throughput(10, 4, 1, 2.0) == 20.0
