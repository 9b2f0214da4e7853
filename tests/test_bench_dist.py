"""The benchmark's multi-replica aggregation (CPU, gloo, world size 2).

Each rank runs its own seeded batch; the job's time is the slowest rank's and
its throughput counts every rank's units.  Runs as two spawned processes on
the CPU with the gloo backend over 127.0.0.1."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, units = bench.job_totals(dist, "cpu", 10.0 + 5.0 * rank,
                                     {"kv_bytes": 1000 * (rank + 1), "seqs": 64})
        q.put((rank, ms, units, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_job_totals_max_time_sum_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, units, env in sorted(results):
        assert ms == 15.0                                   # slowest rank
        assert units == {"kv_bytes": 3000.0, "seqs": 128.0}  # summed over ranks
        assert env == (2, rank, 0)


def test_job_totals_single_process():
    import bench
    assert bench.job_totals(None, "cpu", 3.5, {"kv_bytes": 7}) == (3.5, {"kv_bytes": 7.0})
