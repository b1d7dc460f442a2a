"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the max-over-ranks
timing reduction and the whole-job aggregation used for weak scaling."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, l = bench.dist_env()
    mine = 10.0 + 5.0 * rank  # rank 1 is the slowest
    t = bench.max_over_ranks(mine)
    value, ms = bench.aggregate(t, w, tokens_per_rank_step=1000, steps=4)
    q.put((r, w, t, value, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, t, value, ms in res:
        assert w == 2 and t == 15.0
        assert value == pytest.approx(2 * 1000 * 4 / 0.015)
        assert ms == pytest.approx(15.0 / 4)


def test_aggregate_single_rank():
    v, ms = bench.aggregate(20.0, 1, 16384, 10)
    assert v == pytest.approx(16384 * 10 / 0.02) and ms == 2.0
