"""The bench's multi-rank bookkeeping on CPU: two gloo ranks (one process
each, rendezvous on 127.0.0.1) agree on the slowest rank's time and on the
whole-job throughput. The GPU path runs one replica per rank and has no
data-path collective, so this is all the N > 1 path adds."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.rank_info()
        mine = 0.010 * (rank + 1)                      # rank 1 is the slower one
        slowest = bench.slowest_rank_seconds(torch, mine, world, torch.device("cpu"))
        value = bench.job_value(1_000_000, 100, world, slowest)
        out.put((r, w, lr, slowest, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    assert [(r, w, lr) for r, w, lr, _, _ in results] == [(0, 2, 0), (1, 2, 1)]
    for _, _, _, slowest, value in results:
        assert slowest == pytest.approx(0.020)
        # both ranks' bytes over the slowest rank's time
        assert value == pytest.approx(2 * 1_000_000 * 100 / 0.020 / 1e9)


def test_one_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_seconds(torch, 0.5, 1, torch.device("cpu")) == 0.5
    assert bench.job_value(10, 3, 1, 2.0) == pytest.approx(15 / 1e9)
