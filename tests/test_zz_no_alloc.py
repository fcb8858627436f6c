"""attn_fwd_noalloc: the forward for callers that must not allocate device memory.

Such callers (a process whose device memory belongs to its own allocator, code
held to a fixed device-memory budget, latency-critical paths that may not pay
for cudaMalloc's device-wide synchronisation) use this entry point, which keeps
the kernel's status words in a static device array instead of a cudaMalloc'd
buffer.

The test calls it through the C ABI twice in a row, on different inputs.  It
runs the same kernel with the same grid schedule as attn_fwd, so each result
must equal attn_fwd's bit for bit; each is also compared with the fp64 oracle
at the parity bars of the other GPU tests.  This file is collected last; it
also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_attention_68_gb300 import binding
from exact_attention_68_gb300.workloads import default_scale, make_qkv
from gpu_helpers import compare
from oracle import attention_fwd

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, out, lse, scale, causal):
    B, H, S, D = q.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                lse.data_ptr(), B, H, S, D, scale, 1 if causal else 0, 1, stream)


@pytest.mark.parametrize("shape,causal", [((2, 4, 1000, 128), True), ((1, 3, 777, 64), False)])
def test_noalloc_matches_attn_fwd_two_calls_in_a_row(cuda_device, shape, causal):
    lib = binding.load_library()
    dev = torch.device("cuda:0")
    scale = default_scale(shape[3])
    for seed in (31, 32):  # two calls in a row share the static scratch array
        q_h, k_h, v_h = make_qkv(shape, seed=seed)
        q, k, v = (x.to(dev) for x in (q_h, k_h, v_h))
        ref_out, ref_lse = binding.attn_fwd(q, k, v, scale=scale, causal=causal)
        out = torch.full_like(q, float("nan"))
        lse = torch.full(ref_lse.shape, float("nan"), dtype=torch.float32, device=dev)
        rc = _noalloc(lib, q, k, v, out, lse, scale, causal)
        assert rc == binding.ATTN_OK, binding.AttnError(rc, "attn_fwd_noalloc")
        torch.cuda.synchronize()
        # same kernel, same schedule: bit for bit what attn_fwd wrote
        assert torch.equal(out, ref_out)
        assert torch.equal(lse, ref_lse)
        # and within the parity bars of the fp64 oracle
        ro, rl = attention_fwd(*(x.float().numpy() for x in (q_h, k_h, v_h)), scale, causal)
        compare(out.cpu().double().numpy(), lse.cpu().double().numpy(), ro, rl,
                f"noalloc {shape} causal={causal} seed={seed}")
    assert binding.device_status() == binding.ATTN_OK
