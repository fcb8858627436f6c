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


def test_bench_parity_block_uses_the_oracle_rows():
    """The bench line's parity block: oracle rows against the outputs on the
    same (b, h, row) triples; a planted error in one output row fails it."""
    import numpy as np
    import torch
    import bench
    from exact_attention_68_gb300.workloads import make_qkv
    from oracle import attention_fwd
    q, k, v = make_qkv((1, 2, 64, 16), seed=3)
    qn, kn, vn = bench.as_numpy(q, k, v)
    checked = []
    bench.oracle_rows_sample(qn, kn, vn, 0.25, True, 16, [0, 1], 1e9, checked)
    ro, rl = attention_fwd(qn.astype(np.float64), kn.astype(np.float64), vn.astype(np.float64),
                           0.25, True)
    out = torch.from_numpy(ro).to(torch.bfloat16)
    lse = torch.from_numpy(rl).float()
    res = bench.parity_of_outputs(checked, out, lse)
    assert res["rows"] == 32 and res["pass"], res
    bad = out.clone()
    bad[0, 1, 63, 5] += 0.5  # the last row of head 1 is one of the sampled rows
    assert not bench.parity_of_outputs(checked, bad, lse)["pass"]
