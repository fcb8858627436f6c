"""GPU parity with fp16 inputs (attn_fwd_ex / attn_bwd_ex with ATTN_F16).

The same oracles and bars as the bf16 tests: fp16 has the finer rounding
(unit roundoff 2^-11 against bf16's 2^-8), so the bf16-derived bars hold
with room to spare.  The inputs are the same seeded draws rounded to fp16.
"""
import numpy as np
import pytest
import torch

from exact_attention_68_gb300 import binding
from exact_attention_68_gb300.workloads import WORKLOADS, check_rows, default_scale, make_qkv
from gpu_helpers import bwd_magnitudes, compare, compare_grad, to_f64
from oracle import attention_bwd, attention_fwd, attention_rows

pytestmark = pytest.mark.gpu

F16 = torch.float16


def _fwd(q, k, v, scale, causal):
    out, lse = binding.attn_fwd(*(x.to("cuda:0") for x in (q, k, v)), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    assert out.dtype == F16
    return out.cpu(), lse.cpu()


SHAPES = [(1, 2, 128, 64), (2, 3, 129, 64), (1, 2, 200, 128), (2, 1, 513, 128), (1, 4, 1024, 128),
          (1, 1, 7, 64)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_fp16_forward_full_oracle(cuda_device, shape, causal):
    q, k, v = make_qkv(shape, seed=61, dtype=F16)
    scale = default_scale(shape[3])
    out, lse = _fwd(q, k, v, scale, causal)
    ro, rl = attention_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale, causal)
    compare(to_f64(out), to_f64(lse), ro, rl, f"fp16 {shape} causal={causal}")


@pytest.mark.parametrize("name", ["c3", "c4"])
def test_fp16_forward_workload_rows(cuda_device, name):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w, seed=0, dtype=F16)
    scale = default_scale(w.D)
    out, lse = _fwd(q, k, v, scale, w.causal)
    idx = check_rows(w)
    if name == "c4":  # every row of two heads plus a random sample (fp16 c4 is a second pass)
        rng = np.random.default_rng(62)
        pick = rng.integers(0, idx.shape[0], 4096)
        idx = idx[np.unique(pick)]
    ro, rl = attention_rows(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale,
                            w.causal, idx)
    og = to_f64(out)[idx[:, 0], idx[:, 1], idx[:, 2]]
    lg = to_f64(lse)[idx[:, 0], idx[:, 1], idx[:, 2]]
    compare(og, lg, ro, rl, f"fp16 {name}")


def test_fp16_is_not_read_as_bf16(cuda_device):
    """The same bits as bf16 mean other numbers: the two calls must disagree,
    and only the fp16 one matches the oracle of the fp16 values."""
    q, k, v = make_qkv((1, 2, 256, 64), seed=63, dtype=F16)
    scale = default_scale(64)
    out16, _ = _fwd(q, k, v, scale, True)
    qb, kb, vb = (x.view(torch.bfloat16) for x in (q, k, v))
    outb, _ = binding.attn_fwd(*(x.to("cuda:0") for x in (qb, kb, vb)), scale=scale, causal=True)
    torch.cuda.synchronize()
    binding.device_status()
    assert not torch.equal(out16.view(torch.int16), outb.cpu().view(torch.int16))


@pytest.mark.parametrize("shape", [(1, 2, 128, 64), (2, 2, 300, 128), (1, 2, 513, 64)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_fp16_backward_full_oracle(cuda_device, shape, causal):
    q, k, v = make_qkv(shape, seed=64, dtype=F16)
    g = torch.Generator().manual_seed(65)
    dout = torch.randn(shape, generator=g).to(F16)
    scale = default_scale(shape[3])
    n = [x.double().numpy() for x in (q, k, v, dout)]
    ro, rl = attention_fwd(*n[:3], scale, causal)
    out = torch.from_numpy(ro).to(F16)
    lse = torch.from_numpy(rl).to(torch.float32)
    dev = [x.to("cuda:0") for x in (q, k, v, out, lse, dout)]
    dq, dk, dv, _ = binding.attn_bwd(*dev, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    assert dq.dtype == F16
    rq, rk, rv = attention_bwd(*n, scale, causal)
    B, H, S, _ = shape
    rows = np.arange(S)
    for b in range(B):
        for h in range(H):
            Mq, Mk, Mv = bwd_magnitudes(*n, scale, causal, b, h, rows, rows)
            compare_grad(to_f64(dq.cpu())[b, h], rq[b, h], Mq, f"fp16 dq {shape}")
            compare_grad(to_f64(dk.cpu())[b, h], rk[b, h], Mk, f"fp16 dk {shape}")
            compare_grad(to_f64(dv.cpu())[b, h], rv[b, h], Mv, f"fp16 dv {shape}")


def test_fp16_chained_forward_backward(cuda_device):
    shape = (2, 4, 1024, 128)
    q, k, v = make_qkv(shape, seed=66, dtype=F16)
    g = torch.Generator().manual_seed(67)
    dout = torch.randn(shape, generator=g).to(F16)
    scale = default_scale(128)
    qd, kd, vd, dd = (x.to("cuda:0") for x in (q, k, v, dout))
    out, lse = binding.attn_fwd(qd, kd, vd, scale=scale, causal=True)
    dq, dk, dv, _ = binding.attn_bwd(qd, kd, vd, out, lse, dd, scale=scale, causal=True)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    n = [x.double().numpy() for x in (q, k, v, dout)]
    rq, rk, rv = attention_bwd(*n, scale, True)
    rows = np.arange(shape[2])
    for b, h in ((0, 0), (1, 3)):
        Mq, Mk, Mv = bwd_magnitudes(*n, scale, True, b, h, rows, rows)
        compare_grad(to_f64(dq.cpu())[b, h], rq[b, h], Mq, "fp16 chained dq")
        compare_grad(to_f64(dk.cpu())[b, h], rk[b, h], Mk, "fp16 chained dk")
        compare_grad(to_f64(dv.cpu())[b, h], rv[b, h], Mv, "fp16 chained dv")
