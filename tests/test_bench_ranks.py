"""The benchmark's multi-rank host logic on CPU (gloo, world size 2).

Each rank of `bench.py --gpus N` runs an independent replica; the job's time is
the maximum over ranks and its throughput counts every rank's bytes.  This
checks the reduction and the throughput formula with two gloo processes.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    import torch.distributed as dist
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, lr = bench.dist_env()
    times = [10.0 + 5.0 * rank, 2.0 - rank]          # rank 1 is slower on the first entry
    mx = bench.reduce_over_ranks(times, "max")
    sm = bench.reduce_over_ranks([1.0 + rank], "sum")
    bench.barrier()
    q.put((rank, (w, r, lr), mx, sm))
    dist.destroy_process_group()


def test_two_rank_reduction_and_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, mx, sm in out:
        assert env == (2, rank, rank)
        assert mx == [15.0, 2.0]
        assert sm == [3.0]
    import bench
    # two replicas of 1e9 bytes per step, 4 steps, slowest rank 2 ms -> 4000 GB/s
    assert bench.job_gbs(2, 10 ** 9, 4, 2.0) == pytest.approx(4000.0)


def test_single_process_reduction_is_identity():
    import bench
    assert bench.reduce_over_ranks([1.0, 2.0], "max") == [1.0, 2.0]
