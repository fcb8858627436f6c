"""Failure detection on the GPU without a GPU fault.

A bound of 0 ns on the in-kernel waits makes the first wait that is not
already satisfied run out.  The kernel must record the timeout in the device
status word, let every copy and MMA it started finish, free its tensor memory
and return; the context stays usable and the next normal call is correct.
"""
import pytest
import torch

from exact_attention_68_gb300 import binding
from exact_attention_68_gb300.workloads import default_scale, make_qkv
from gpu_helpers import compare, run_gpu, to_f64
from oracle import attention_fwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
def test_forced_wait_timeout_reports_and_recovers(cuda_device, D):
    q, k, v = make_qkv((2, 2, 1024, D), seed=21)
    dev = torch.device("cuda:0")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    assert binding.device_status() == binding.ATTN_OK
    binding.attn_fwd_bounded(qd, kd, vd, causal=True, wait_timeout_ns=0)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_ERR_TIMEOUT
    # the status word was cleared by the read, and the GPU still computes correctly
    assert binding.device_status() == binding.ATTN_OK
    out, lse = run_gpu(q, k, v, default_scale(D), True)
    ro, rl = attention_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                           default_scale(D), True)
    compare(to_f64(out), to_f64(lse), ro, rl, "after timeout")


def test_generous_bound_does_not_time_out(cuda_device):
    q, k, v = (x.to("cuda:0") for x in make_qkv((1, 8, 4096, 128), seed=22))
    binding.attn_fwd_bounded(q, k, v, causal=True, wait_timeout_ns=10_000_000_000)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK


def test_argument_errors_on_gpu_launch_nothing(cuda_device):
    q, k, v = (x.to("cuda:0") for x in make_qkv((1, 1, 128, 64)))
    out = torch.full_like(q, 7.0)
    lse = torch.full((1, 1, 128), 7.0, device="cuda:0")
    lib = binding.load_library()
    rc = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                      1, 1, 128, 100, 0.1, 1, None)
    assert rc == binding.ATTN_ERR_UNSUPPORTED
    rc = lib.attn_fwd(q.data_ptr() + 2, k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                      1, 1, 128, 64, 0.1, 1, None)
    assert rc == binding.ATTN_ERR_MISALIGNED
    torch.cuda.synchronize()
    assert (out == 7.0).all() and (lse == 7.0).all()


@pytest.mark.parametrize("D", [64, 128])
def test_bwd_forced_wait_timeout_reports_and_recovers(cuda_device, D):
    shape = (2, 2, 1024, D)
    q, k, v = (x.to("cuda:0") for x in make_qkv(shape, seed=23))
    out, lse = binding.attn_fwd(q, k, v, causal=True)
    dout = torch.ones_like(q)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    binding.attn_bwd_bounded(q, k, v, out, lse, dout, causal=True, wait_timeout_ns=0)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_ERR_TIMEOUT
    assert binding.device_status() == binding.ATTN_OK
    # the next normal call runs to completion
    dq, dk, dv, _ = binding.attn_bwd(q, k, v, out, lse, dout, causal=True)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    assert all(torch.isfinite(t.float()).all() for t in (dq, dk, dv))
