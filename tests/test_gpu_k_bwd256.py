"""GPU parity of the backward for head dimensions above 128 (the kernels 256
columns wide) against the fp64 gradient oracle.

Widths other than 256 (136, 192, 200) run on the same kernels with the
columns past D read as zero and never stored.  Each gradient sits in front of
a sentinel guard that must stay untouched.  The element-wise bar is the one
the other backward tests use (2^-7 of the magnitude the element accumulates,
plus 1e-6; relative Frobenius error <= 2^-7 per tensor).
"""
import numpy as np
import pytest
import torch

from exact_attention_68_gb300 import binding
from exact_attention_68_gb300.workloads import default_scale, make_qkv
from gpu_helpers import bwd_magnitudes, compare_grad, run_gpu, to_f64
from oracle import attention_bwd, attention_bwd_rows, attention_fwd

pytestmark = pytest.mark.gpu

SENTINEL = 7.0
GUARD = 4096


def _guarded(shape, dtype):
    n = int(np.prod(shape))
    buf = torch.full((n + GUARD,), SENTINEL, dtype=dtype, device="cuda:0")
    return buf, buf[:n].view(shape)


def _dout(shape, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(dtype)


def _bwd_vs_oracle(shape, causal, seed, dtype=torch.bfloat16, scale=None):
    B, H, S, D = shape
    q, k, v = make_qkv(shape, seed=seed, dtype=dtype)
    dout = _dout(shape, seed + 1, dtype)
    scale = default_scale(D) if scale is None else scale
    n = [x.double().numpy() for x in (q, k, v, dout)]
    ro, rl = attention_fwd(*n[:3], scale, causal)
    out = torch.from_numpy(ro).to(dtype)
    lse = torch.from_numpy(rl).to(torch.float32)
    dev = [x.to("cuda:0") for x in (q, k, v, out, lse, dout)]
    bufs = [_guarded(shape, dtype) for _ in range(3)]
    dbuf, delta = _guarded(shape[:3], torch.float32)
    dq, dk, dv, _ = binding.attn_bwd(*dev, scale=scale, causal=causal, dq=bufs[0][1],
                                     dk=bufs[1][1], dv=bufs[2][1], delta=delta)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    for buf, t in bufs:
        assert (buf[t.numel():] == SENTINEL).all(), "the backward wrote past the end of a gradient"
    assert (dbuf[delta.numel():] == SENTINEL).all()
    rq, rk, rv = attention_bwd(*n, scale, causal)
    rows = np.arange(S)
    for b in range(B):
        for h in range(H):
            Mq, Mk, Mv = bwd_magnitudes(*n, scale, causal, b, h, rows, rows)
            compare_grad(to_f64(dq)[b, h], rq[b, h], Mq, f"{shape} dq b{b}h{h}")
            compare_grad(to_f64(dk)[b, h], rk[b, h], Mk, f"{shape} dk b{b}h{h}")
            compare_grad(to_f64(dv)[b, h], rv[b, h], Mv, f"{shape} dv b{b}h{h}")
    ref_delta = (dout.double() * out.double()).sum(-1).numpy()
    np.testing.assert_allclose(to_f64(delta), ref_delta, rtol=1e-5, atol=1e-5)
    return dq, dk, dv


@pytest.mark.parametrize("D", [136, 192, 200, 256])
@pytest.mark.parametrize("S", [1, 129, 201])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_bwd_wide_heads_full_oracle(cuda_device, D, S, causal):
    _bwd_vs_oracle((2, 2, S, D), causal, seed=300 + D + S)


def test_bwd_d256_peaked_softmax_other_scale(cuda_device):
    for causal in (True, False):
        _bwd_vs_oracle((1, 2, 384, 256), causal, seed=331, scale=0.11)


def test_bwd_d256_fp16(cuda_device):
    _bwd_vs_oracle((1, 2, 300, 256), True, seed=341, dtype=torch.float16)


def test_bwd_d256_deterministic(cuda_device):
    shape = (1, 3, 700, 256)
    q, k, v = (x.to("cuda:0") for x in make_qkv(shape, seed=351))
    dout = _dout(shape, 352).to("cuda:0")
    out, lse = binding.attn_fwd(q, k, v, causal=True)
    a = binding.attn_bwd(q, k, v, out, lse, dout, causal=True)
    b = binding.attn_bwd(q, k, v, out, lse, dout, causal=True)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("D", [256, 192])
def test_bwd_wide_heads_chained_long(cuda_device, D):
    """fwd → bwd on the GPU at S = 4096, sampled rows of two heads."""
    shape = (1, 3, 4096, D)
    q, k, v = make_qkv(shape, seed=360 + D)
    dout = _dout(shape, 361 + D)
    scale = default_scale(D)
    out, lse = run_gpu(q, k, v, scale, True)
    dev = [x.to("cuda:0") for x in (q, k, v, out, lse, dout)]
    dq, dk, dv, _ = binding.attn_bwd(*dev, scale=scale, causal=True)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    n = [x.float().numpy() for x in (q, k, v, dout)]
    rng = np.random.default_rng(362)
    rows = np.unique(np.concatenate([[0, 63, 64, 127, 128, 4095], rng.integers(0, 4096, 90)]))
    for h in (0, 2):
        rq, rk, rv = attention_bwd_rows(*n, scale, True, 0, h, rows, rows)
        Mq, Mk, Mv = bwd_magnitudes(*n, scale, True, 0, h, rows, rows)
        compare_grad(to_f64(dq.cpu())[0, h, rows], rq, Mq, f"D={D} dq h{h}")
        compare_grad(to_f64(dk.cpu())[0, h, rows], rk, Mk, f"D={D} dk h{h}")
        compare_grad(to_f64(dv.cpu())[0, h, rows], rv, Mv, f"D={D} dv h{h}")
