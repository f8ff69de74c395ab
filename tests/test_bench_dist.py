"""bench.py's multi-rank path on CPU: two gloo ranks, each an independent
replica; the job's time is the slowest rank's and its units are the sum."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    w, r, _ = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    seconds, units = bench.aggregate(1.5 + rank, 64.0 * (rank + 1), dist)
    q.put((r, seconds, units))
    dist.destroy_process_group()


def test_two_rank_aggregate_takes_max_time_and_total_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5, 192.0), (1, 2.5, 192.0)]


def test_single_rank_aggregate_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.aggregate(2.0, 64.0, None) == (2.0, 64.0)
