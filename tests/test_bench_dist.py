"""bench.py's multi-rank host logic on CPU: gloo, world_size 2, 127.0.0.1.

Each rank of a replicated run times its own replica; bench.py brackets the
timed region with barriers and reports the max over ranks.  Here two gloo
ranks feed different times into the same reduction and both must see the max.
"""
import os
import socket

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    got = bench.reduce_max(10.0 + 5.0 * r, w, "cpu")
    bench.barrier(w)
    q.put((r, w, got))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 15.0), (1, 2, 15.0)]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.reduce_max(3.5, 1, "cpu") == 3.5
