"""Multi-process host logic of bench.py's replica mode (world size 2, gloo, CPU only).

bench.py --gpus N runs N independent replicas (the GEMV shards by output rows, but every run
here has one GPU, so there is no collective on the data path): every rank times its own
steps, the step time is the maximum over ranks, and the whole-job value is all ranks' work
over that time.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + 5.0 * rank, 3.0 - rank]  # rank 1 is slower on the first, faster on the second
        got = bench.max_over_ranks(mine, "cpu", world)
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_replica_rate_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(out.get(timeout=10) for _ in range(world))
    assert res[0] == res[1] == [15.0, 3.0]  # element-wise maximum over the ranks, on every rank
    sys.path.insert(0, ROOT)
    import bench
    # 2 replicas x 28 MB of weights each over the slowest rank's 15 ms step
    assert bench.replica_rate(world, 28e6, 15.0) == pytest.approx(2 * 28e6 / 15e-3)


def test_single_process_keeps_values():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], "cpu", 1) == [1.5, 2.5]
    assert bench.replica_rate(1, 1e9, 1000.0) == pytest.approx(1e9)
