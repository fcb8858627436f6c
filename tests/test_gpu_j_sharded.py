"""The head-sharded forward (attn_fwd_sharded) on the GPU.

Every run here has one GPU, so the shards of a multi-process split are run
one after another in one process on cuda:0, each as its rank would: only its
slices are copied to the device and attn_fwd runs on them.  Each shard is
compared with the fp64 oracle on its slices, and bit for bit with the same
slices of the unsharded forward (a slice's result depends only on its own
rows, not on the grid it ran in).
"""
import numpy as np
import pytest
import torch

from exact_attention_68_gb300 import binding
from exact_attention_68_gb300.workloads import default_scale, make_qkv
from gpu_helpers import compare
from oracle import attention_fwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,world,causal", [((2, 4, 1000, 128), 2, True),
                                                ((1, 5, 640, 64), 2, False),
                                                ((1, 5, 300, 128), 3, True),
                                                ((1, 2, 256, 64), 4, True)])
def test_shards_match_the_oracle_and_the_whole_forward(cuda_device, shape, world, causal):
    B, H, S, D = shape
    scale = default_scale(D)
    q, k, v = make_qkv(shape, seed=23)
    whole_out, whole_lse = binding.attn_fwd(*(x.to(cuda_device) for x in (q, k, v)), scale=scale,
                                            causal=causal)
    ro, rl = attention_fwd(*(x.float().numpy() for x in (q, k, v)), scale, causal)
    ro, rl = ro.reshape(B * H, S, D), rl.reshape(B * H, S)
    seen = 0
    for rank in range(world):
        first, count, out, lse = binding.attn_fwd_sharded(q, k, v, scale=scale, causal=causal,
                                                          rank=rank, world=world,
                                                          device=cuda_device)
        torch.cuda.synchronize()
        assert first == seen
        seen += count
        assert out.shape == (count, S, D) and lse.shape == (count, S)
        if count == 0:
            continue
        compare(out.cpu().double().numpy(), lse.cpu().double().numpy(),
                ro[first:first + count], rl[first:first + count],
                f"shard {rank}/{world} of {shape}")
        assert torch.equal(out, whole_out.view(B * H, S, D)[first:first + count])
        assert torch.equal(lse, whole_lse.view(B * H, S)[first:first + count])
    assert seen == B * H
    assert binding.device_status() == binding.ATTN_OK
