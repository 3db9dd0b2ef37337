"""World-size-2 check (gloo, CPU) of the benchmark's multi-replica timing: every rank
reports its own elapsed time, the job time is the max over ranks, and the whole-job
throughput counts the tokens of all ranks ("replicas only": no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    d = bench.Dist("gloo")
    d.barrier()
    elapsed = 1.0 + rank          # rank 1 is the slow one
    job = d.max(elapsed)
    tokens_per_rank = 8 * 10
    value = tokens_per_rank * d.world / job
    q.put((rank, job, value))
    d.close()


def test_two_rank_max_timing_and_aggregate_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, job, value in res:
        assert job == 2.0
        assert value == pytest.approx(80.0)
