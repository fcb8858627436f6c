"""The head-sharded split of one forward over processes (one per GPU), on CPU.

attn_shard_range (C ABI) gives each rank a contiguous range of the B·H
(batch, head) slices; every slice is independent (FlashAttention-2 blog,
"FlashAttention-2 Optimizations" §3: parallel over batch and heads), so the
ranks exchange nothing.  Checked here: the ranges partition the slices in
order and evenly, bad arguments are refused, a rank's slices of a contiguous
[B, H, S, D] tensor are the contiguous block the binding hands to attn_fwd,
and two gloo ranks that each compute their share (with the fp64 oracle
standing in for the GPU kernel, on CPU) reassemble the whole forward.
"""
import ctypes
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from exact_attention_68_gb300 import binding
from exact_attention_68_gb300.build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return binding.load_library(build_library())


@pytest.mark.parametrize("units", [0, 1, 2, 5, 31, 32, 33, 128, 1000])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 7, 8, 64])
def test_ranges_partition_the_slices_in_order(lib, units, world):
    ranges = [binding.shard_range(units, world, r) for r in range(world)]
    assert ranges[0][0] == 0
    for (f0, c0), (f1, _) in zip(ranges, ranges[1:]):
        assert f0 + c0 == f1  # contiguous, in rank order
    assert ranges[-1][0] + ranges[-1][1] == units  # every slice once
    counts = [c for _, c in ranges]
    assert max(counts) - min(counts) <= 1  # even
    assert counts == sorted(counts, reverse=True)  # the extra slices go to the first ranks
    assert sum(counts) == units


def test_bad_arguments_are_refused(lib):
    f, c = ctypes.c_int64(-7), ctypes.c_int64(-7)
    for units, world, rank in ((-1, 2, 0), (4, 0, 0), (4, 2, 2), (4, 2, -1)):
        rc = lib.attn_shard_range(units, world, rank, ctypes.byref(f), ctypes.byref(c))
        assert rc == binding.ATTN_ERR_INVALID_ARG
        assert (f.value, c.value) == (-7, -7)  # outputs untouched
    assert lib.attn_shard_range(4, 2, 0, None, ctypes.byref(c)) == binding.ATTN_ERR_INVALID_ARG
    with pytest.raises(binding.AttnError):
        binding.shard_range(4, 2, 5)


def test_a_ranks_slices_are_one_contiguous_block():
    B, H, S, D = 3, 5, 16, 8
    t = torch.arange(B * H * S * D, dtype=torch.float32).view(B, H, S, D).to(torch.bfloat16)
    for world in (2, 4, 6):
        for rank in range(world):
            first, count = binding.shard_range(B * H, world, rank)
            block = t.view(B * H, S, D)[first:first + count]
            assert block.is_contiguous()
            assert block.data_ptr() == t.data_ptr() + first * S * D * t.element_size()
            for n in range(count):
                b, h = divmod(first + n, H)
                assert torch.equal(block[n], t[b, h])


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, shape, q_out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    from exact_attention_68_gb300 import binding as bd
    from exact_attention_68_gb300.workloads import make_qkv
    from oracle import attention_fwd
    dist.init_process_group("gloo", rank=rank, world_size=world)
    B, H, S, D = shape
    q, k, v = make_qkv(shape, seed=9)  # every rank draws the same whole problem
    first, count = bd.shard_range(B * H, world, rank)
    part = [t.view(B * H, S, D)[first:first + count].float().numpy()[None] for t in (q, k, v)]
    out, lse = attention_fwd(*part, 0.3, True)  # stands in for this rank's GPU kernel
    got = [None] * world
    dist.all_gather_object(got, (first, count, out[0], lse[0]))
    if rank == 0:
        full_out = np.concatenate([g[2] for g in sorted(got, key=lambda g: g[0])])
        full_lse = np.concatenate([g[3] for g in sorted(got, key=lambda g: g[0])])
        ro, rl = attention_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), 0.3, True)
        q_out.put((sorted((g[0], g[1]) for g in got),
                   bool(np.array_equal(full_out.reshape(ro.shape), ro)),
                   bool(np.array_equal(full_lse.reshape(rl.shape), rl))))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reassemble_the_whole_forward():
    shape = (3, 3, 40, 8)  # 9 slices: ranks take 5 and 4
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, shape, q)) for r in range(2)]
    for p in procs:
        p.start()
    ranges, out_equal, lse_equal = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert ranges == [(0, 5), (5, 4)]
    assert out_equal and lse_equal
