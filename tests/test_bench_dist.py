"""The bench's multi-rank host logic on CPU: world size 2 over gloo (no GPU).

The decode step does not shard (each GPU runs independent sessions on its own
replica), so the only cross-rank work is the barrier and the job aggregate:
units summed over ranks divided by the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    t, u = bench.reduce_job(w, elapsed_s=1.0 + rank, units=10.0 * (rank + 1))
    q.put((r, w, t, u))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_job_aggregate_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for r, w, t, u in res:
        assert w == 2 and t == 2.0 and u == 30.0  # max time, summed units


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_job(1, 3.5, 7) == (3.5, 7)
