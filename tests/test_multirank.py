"""The multi-rank host path of bench.py on CPU: two processes on the gloo
backend (one process per GPU is the launch form; here no GPU is involved)
set up the process group, meet at the barriers that bracket the timed region
and agree on the slowest rank's time (the reported value is the max over
ranks).  The library's path does not shard across GPUs ("replicas only"), so
this is the whole N > 1 logic."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    ws, r, local = bench.dist_setup(world)
    assert (ws, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(ws)
    got = bench.max_over_ranks(ws, 10.0 * (rank + 1))   # rank 1 is the slowest
    bench.barrier(ws)
    dist.destroy_process_group()
    q.put((rank, got))


def test_two_gloo_ranks_barrier_and_max():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 20.0, 1: 20.0}
