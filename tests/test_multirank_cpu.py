"""The multi-rank bench path on CPU: two gloo ranks run independent replicas and
the whole-job rate uses the slowest rank's time (no GPU)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    import torch
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)

    def max_over_ranks(x):
        t = torch.tensor([x], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    elapsed = 1.0 + rank          # rank 1 is the slow one: 2 s
    rate, t = bench.aggregate(elapsed, 100.0, ws, max_over_ranks)
    dist.barrier()
    q.put((rank, rate, t))
    dist.destroy_process_group()


def test_two_rank_aggregate_takes_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, rate, t in out:
        assert t == pytest.approx(2.0)          # max over ranks
        assert rate == pytest.approx(2 * 100.0 / 2.0)


def test_single_rank_aggregate():
    import bench
    rate, t = bench.aggregate(0.5, 10.0, 1)
    assert (rate, t) == (20.0, 0.5)
