"""The multi-GPU path of bench.py is N independent replicas; its host logic
(max of the per-rank times, sum of the per-rank work) is checked here with
two gloo processes on CPU."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    d = bench._init_pg(world)
    t, u = bench.aggregate(0.5 + rank, 100.0 * (rank + 1), d)
    q.put((rank, t, u))
    d.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for _, t, u in res:
        assert t == pytest.approx(1.5)     # slowest rank
        assert u == pytest.approx(300.0)   # all ranks' work


def test_aggregate_single_process_is_identity():
    import bench
    assert bench.aggregate(0.25, 7.0, None) == (0.25, 7.0)
