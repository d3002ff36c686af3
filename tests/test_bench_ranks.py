"""bench.py's multi-rank aggregation on two CPU ranks (gloo). Requests are
independent, so N GPUs run N replicas with no exchange; the job's time for the
timed steps is the slowest rank's, and the job rate counts every rank's rounds."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q) -> None:
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    def max_over_ranks(v):
        t = torch.tensor([v], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    dist.barrier()
    # rank r spends (r + 1) ms per step over 10 steps
    value, ms = bench.job_rate(10.0 * (rank + 1), 10, world, max_over_ranks)
    q.put((rank, value, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_report_the_slowest_rank():
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
    assert [r for r, _, _ in out] == [0, 1]
    for _, value, ms in out:
        assert ms == 2.0                 # the slower rank's 2 ms per step
        assert value == 2 * 1e3 / 2.0    # both replicas' rounds over that time


def test_one_rank_needs_no_reduction():
    import bench
    value, ms = bench.job_rate(50.0, 10, 1)
    assert ms == 5.0 and value == 200.0
