"""GPU checks of the Python-level API: the autograd wrapper and CUDA-graph
capture of the C entry points (no host synchronisation inside them)."""
import numpy as np
import pytest
import torch

from exact_attention_68_gb300 import binding
from exact_attention_68_gb300.workloads import default_scale, make_qkv
from gpu_helpers import bwd_magnitudes, compare_grad, to_f64
from oracle import attention_bwd, attention_fwd

pytestmark = pytest.mark.gpu


def test_autograd_wrapper_matches_the_oracle(cuda_device):
    shape = (1, 2, 300, 128)
    q, k, v = make_qkv(shape, seed=81)
    g = torch.Generator().manual_seed(82)
    dout = torch.randn(shape, generator=g).to(torch.bfloat16)
    scale = default_scale(128)
    qd, kd, vd = (x.to("cuda:0").requires_grad_(True) for x in (q, k, v))
    out = binding.attention(qd, kd, vd, scale=scale, causal=True)
    out.backward(dout.to("cuda:0"))
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    n = [x.float().numpy() for x in (q, k, v, dout)]
    ro, _ = attention_fwd(*n[:3], scale, True)
    err = np.abs(to_f64(out.detach().cpu()) - ro)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    rq, rk, rv = attention_bwd(*n, scale, True)
    rows = np.arange(shape[2])
    for h in range(shape[1]):
        Mq, Mk, Mv = bwd_magnitudes(*n, scale, True, 0, h, rows, rows)
        compare_grad(to_f64(qd.grad.cpu())[0, h], rq[0, h], Mq, "autograd dq")
        compare_grad(to_f64(kd.grad.cpu())[0, h], rk[0, h], Mk, "autograd dk")
        compare_grad(to_f64(vd.grad.cpu())[0, h], rv[0, h], Mv, "autograd dv")


def test_forward_and_backward_replay_in_a_cuda_graph(cuda_device):
    """Captured once, replayed on new inputs: bitwise the eager results."""
    shape = (2, 4, 1024, 128)
    scale = default_scale(128)
    dev = torch.device("cuda:0")
    q, k, v = (x.to(dev) for x in make_qkv(shape, seed=83))
    dout = torch.randn(shape, device=dev).to(torch.bfloat16)
    out, lse = binding.attn_fwd(q, k, v, scale=scale, causal=True)   # first call: set-up
    dq, dk, dv, delta = binding.attn_bwd(q, k, v, out, lse, dout, scale=scale, causal=True)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            binding.attn_fwd(q, k, v, scale=scale, causal=True, out=out, lse=lse)
            binding.attn_bwd(q, k, v, out, lse, dout, scale=scale, causal=True, dq=dq, dk=dk,
                             dv=dv, delta=delta)
    torch.cuda.current_stream(dev).wait_stream(side)
    q2, k2, v2 = (x.to(dev) for x in make_qkv(shape, seed=84))
    q.copy_(q2), k.copy_(k2), v.copy_(v2)
    graph.replay()
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    ref_out, ref_lse = binding.attn_fwd(q2, k2, v2, scale=scale, causal=True)
    ref = binding.attn_bwd(q2, k2, v2, ref_out, ref_lse, dout, scale=scale, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    for a, b in zip((dq, dk, dv, delta), ref):
        assert torch.equal(a, b)


def test_entry_points_from_a_fresh_host_thread(cuda_device):
    """A thread that has made no CUDA runtime call of its own (as autograd's
    worker threads may be): forward, backward and the allocation-free forward
    all bind the device's context themselves."""
    import threading
    shape = (1, 2, 256, 64)
    dev = torch.device("cuda:0")
    q, k, v = (x.to(dev) for x in make_qkv(shape, seed=85))
    dout = torch.ones_like(q)
    ref_out, ref_lse = binding.attn_fwd(q, k, v, causal=True)
    ref_grads = binding.attn_bwd(q, k, v, ref_out, ref_lse, dout, causal=True)
    torch.cuda.synchronize()
    lib = binding.load_library()
    res = {}

    def worker():
        try:
            out = torch.empty_like(q)
            lse = torch.empty_like(ref_lse)
            # raw C calls on the legacy default stream, so no torch call binds the thread first
            rc1 = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               lse.data_ptr(), 1, 2, 256, 64, 0.125, 1, None)
            g = [torch.empty_like(q) for _ in range(3)] + [torch.empty_like(ref_lse)]
            rc2 = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               lse.data_ptr(), dout.data_ptr(), *(t.data_ptr() for t in g),
                               1, 2, 256, 64, 0.125, 1, None)
            rc3 = lib.attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                       lse.data_ptr(), 1, 2, 256, 64, 0.125, 1, 1, None)
            res["rc"] = (rc1, rc2, rc3)
            res["out"], res["lse"], res["grads"] = out, lse, g
        except Exception as e:  # reported below
            res["exc"] = e

    th = threading.Thread(target=worker)
    th.start()
    th.join()
    assert "exc" not in res, res.get("exc")
    torch.cuda.synchronize()
    assert res["rc"] == (0, 0, 0), res["rc"]
    assert torch.equal(res["out"], ref_out) and torch.equal(res["lse"], ref_lse)
    for a, b in zip(res["grads"], ref_grads):
        assert torch.equal(a, b)
