"""The multi-rank bench path on CPU: two gloo ranks run independent replicas and
the whole-job rate uses the slowest rank's time (no GPU)."""
import json
import os
import socket
import subprocess

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


def test_bench_launcher_runs_two_replicas_through_its_rank_flow():
    """bench.launch_replicas starts two processes through torch.distributed.run; each
    runs bench's rank flow (barrier, timed steps, barrier, max over ranks) around a host
    stand-in step, rank 1 twice as slow; rank 0 alone prints one line with n_gpus = 2
    and the rate over the slowest rank's time."""
    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = bench.launch_replicas(2, [], script=os.path.join(root, "tests", "replica_standin.py"),
                              stdout=subprocess.PIPE)
    assert r.returncode == 0
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2
    assert d["elapsed_s"] >= d["steps"] * 0.04 * 0.99   # rank 1's 5 x 40 ms
    assert d["value"] == pytest.approx(2 * 100.0 * d["steps"] / d["elapsed_s"])


def test_single_rank_replica_rate():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    ranks = bench.Ranks("gloo")
    n = []
    rate, t = bench.replica_rate(ranks, lambda: n.append(1), 3, 10.0, bench.WallClock())
    assert len(n) == 3 and rate == pytest.approx(30.0 / t)
