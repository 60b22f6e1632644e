"""The multi-rank side of bench.py, on CPU with two gloo ranks (replicas only: no data-path collective).

Each rank times the same workload on its own GPU; the line reports the units all ranks processed
over the slowest rank's time. Here two processes stand in for the ranks with made-up times: the
max-over-ranks helper must return the slower time on every rank, the aggregate must count both
ranks' work, and the reference arm must print on rank 0 only.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(mine, world)
        value = bench.whole_job_value("decode_2112", 1e6, 100, world, slowest)
        args = type("A", (), {"config": "tiny", "steps": 1, "warmup": 0, "ref_seconds": 0.05})()
        ref = bench.run_reference(args, rank, world)
        out.put((rank, slowest, value, ref is None))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_units():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, ref_none in res:
        assert slowest == 15.0                      # both ranks see the slower rank's time
        assert value == pytest.approx(1e6 * 100 * 2 / 1e9 / 0.015)  # both ranks' units over it
        assert ref_none == (rank != 0)              # the reference arm prints on rank 0 only


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_value("prefill", 2e12, 10, 1, 1000.0) == pytest.approx(20.0)
