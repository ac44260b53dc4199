"""The bench's multi-rank bookkeeping on CPU ranks (gloo, world size 2).

Every rank runs its own replica of the step on its own GPU; the job's time is
the slowest rank's, and the job's throughput counts the bytes of all ranks.
Two CPU processes stand in for two GPUs: each reports a different step time,
and both must arrive at the same maximum and the same whole-job figure.
"""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(0.010 * (rank + 1), world, "cpu")
        v = bench.job_throughput(2.0e9, world, t)
        dist.barrier()
        q.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_both_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in procs)
    for rank, t, v in got:
        assert t == 0.020, (rank, t)                  # the slower rank's 20 ms
        assert abs(v - 2 * 2.0e9 / 0.020 / 1e9) < 1e-9, (rank, v)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5, 1, "cpu") == 0.5
    assert bench.job_throughput(1.0e9, 1, 0.5) == 2.0
