"""The N > 1 path of bench.py (replicas only: independent batches, no data-path
collective), run as two gloo ranks on the CPU: the timing is the slowest
rank's, every rank sees it, each rank draws its own batch, and the job rate
counts every replica's tokens."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slower replica
        dist.barrier()
        slowest = bench.max_over_ranks(dist, local_ms, "cpu")
        q.put((rank, slowest, bench.replica_seed(7, rank)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [15.0, 15.0]       # both ranks see the max
    assert got[0][2] != got[1][2]                    # independent batches


def test_job_rate_and_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.5, "cpu") == 3.5
    assert bench.replica_seed(7, 0) == 7
    # 2 replicas x 64 sequences x 100 steps in 20 ms (slowest replica)
    assert bench.job_tokens_per_s(2, 64, 100, 20.0) == 2 * 64 * 100 / 0.020
