"""GPU parity of head dimensions other than 64, 128 and 256 against the fp64
oracle.  They run on the kernel of the next width up (64, 128 or 256
columns; the forward also has 192) with the columns past D read as zero by
TMA and never stored; the
tests check the results against the oracle with the same bars as the native
widths, and that nothing past the end of each output tensor is written."""
import numpy as np
import pytest
import torch

from exact_attention_68_gb300 import binding
from exact_attention_68_gb300.workloads import default_scale, make_qkv
from gpu_helpers import bwd_magnitudes, compare, compare_grad, run_gpu, to_f64
from oracle import attention_bwd, attention_fwd, attention_rows, attention_bwd_rows

pytestmark = pytest.mark.gpu

SENTINEL = 7.0
GUARD = 4096  # elements of sentinel after each output


def _guarded(shape, dtype, device="cuda:0"):
    """A contiguous tensor of `shape` at the front of a buffer whose tail holds SENTINEL."""
    n = int(np.prod(shape))
    buf = torch.full((n + GUARD,), SENTINEL, dtype=dtype, device=device)
    return buf, buf[:n].view(shape)


def _fwd_guarded(q, k, v, scale, causal):
    qd, kd, vd = (x.to("cuda:0") for x in (q, k, v))
    B, H, S, _ = q.shape
    obuf, out = _guarded(q.shape, q.dtype)
    lbuf, lse = _guarded((B, H, S), torch.float32)
    binding.attn_fwd(qd, kd, vd, scale=scale, causal=causal, out=out, lse=lse)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    n = out.numel()
    assert (obuf[n:] == SENTINEL).all(), "the forward wrote past the end of out"
    assert (lbuf[lse.numel():] == SENTINEL).all(), "the forward wrote past the end of lse"
    return out.cpu(), lse.cpu()


# widths below 64 run on the 64-column kernel, 72..120 on the 128-column one,
# 136..248 on the 256-column one
D_FWD = [8, 16, 32, 40, 48, 56, 72, 80, 96, 112, 120, 136, 160, 192, 200, 224, 248]
SHAPES = [(1, 1, 1), (1, 2, 63), (2, 1, 129), (1, 2, 300)]


@pytest.mark.parametrize("D", D_FWD)
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_fwd_head_dims_full_oracle(cuda_device, D, causal):
    for B, H, S in SHAPES:
        shape = (B, H, S, D)
        q, k, v = make_qkv(shape, seed=100 + D)
        scale = default_scale(D)
        out, lse = _fwd_guarded(q, k, v, scale, causal)
        ro, rl = attention_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale, causal)
        compare(to_f64(out), to_f64(lse), ro, rl, f"D={D} {shape} causal={causal}")


@pytest.mark.parametrize("D", [32, 96, 192])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_fwd_head_dims_fp16_and_peaked(cuda_device, D, causal):
    shape = (2, 2, 517, D)
    scale = default_scale(D)
    q, k, v = make_qkv(shape, seed=110 + D, dtype=torch.float16)
    out, lse = _fwd_guarded(q, k, v, scale, causal)
    assert out.dtype == torch.float16
    ro, rl = attention_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale, causal)
    compare(to_f64(out), to_f64(lse), ro, rl, f"fp16 D={D} causal={causal}")
    # q, k ~ N(0, 3^2): rows' running max moves, so the O correction path runs
    q, k, v = make_qkv(shape, seed=120 + D, qk_std=3.0)
    out, lse = _fwd_guarded(q, k, v, scale, causal)
    ro, rl = attention_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale, causal)
    compare(to_f64(out), to_f64(lse), ro, rl, f"peaked D={D} causal={causal}")


@pytest.mark.parametrize("D", [96, 160])
def test_fwd_head_dims_long_sequence_sampled_rows(cuda_device, D):
    B, H, S = 2, 4, 8192
    q, k, v = make_qkv((B, H, S, D), seed=130 + D)
    scale = default_scale(D)
    out, lse = run_gpu(q, k, v, scale, True)
    rng = np.random.default_rng(131)
    idx = np.stack([rng.integers(0, B, 300), rng.integers(0, H, 300), rng.integers(0, S, 300)], 1)
    idx = np.concatenate([idx, [[b, h, r] for b in range(B) for h in range(H)
                                for r in (0, 127, 128, S - 1)]]).astype(np.int64)
    ro, rl = attention_rows(q.float().numpy(), k.float().numpy(), v.float().numpy(), scale, True, idx)
    og = to_f64(out)[idx[:, 0], idx[:, 1], idx[:, 2]]
    lg = to_f64(lse)[idx[:, 0], idx[:, 1], idx[:, 2]]
    compare(og, lg, ro, rl, f"D={D} S=8192")


def _dout(shape, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(dtype)


@pytest.mark.parametrize("D", [8, 32, 40, 72, 96, 120])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_bwd_head_dims_full_oracle(cuda_device, D, causal):
    shape = (2, 2, 201, D)
    q, k, v = make_qkv(shape, seed=140 + D)
    dout = _dout(shape, 141 + D)
    scale = default_scale(D)
    n = [x.double().numpy() for x in (q, k, v, dout)]
    ro, rl = attention_fwd(*n[:3], scale, causal)
    out = torch.from_numpy(ro).to(torch.bfloat16)
    lse = torch.from_numpy(rl).to(torch.float32)
    dev = [x.to("cuda:0") for x in (q, k, v, out, lse, dout)]
    bufs = [_guarded(shape, torch.bfloat16) for _ in range(3)]
    dbuf, delta = _guarded(shape[:3], torch.float32)
    dq, dk, dv, _ = binding.attn_bwd(*dev, scale=scale, causal=causal, dq=bufs[0][1],
                                     dk=bufs[1][1], dv=bufs[2][1], delta=delta)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    for buf, t in bufs:
        assert (buf[t.numel():] == SENTINEL).all(), "the backward wrote past the end of a gradient"
    assert (dbuf[delta.numel():] == SENTINEL).all()
    rq, rk, rv = attention_bwd(*n, scale, causal)
    rows = np.arange(shape[2])
    for b in range(shape[0]):
        for h in range(shape[1]):
            Mq, Mk, Mv = bwd_magnitudes(*n, scale, causal, b, h, rows, rows)
            compare_grad(to_f64(dq)[b, h], rq[b, h], Mq, f"D={D} dq b{b}h{h}")
            compare_grad(to_f64(dk)[b, h], rk[b, h], Mk, f"D={D} dk b{b}h{h}")
            compare_grad(to_f64(dv)[b, h], rv[b, h], Mv, f"D={D} dv b{b}h{h}")
    ref_delta = (dout.double() * out.double()).sum(-1).numpy()
    np.testing.assert_allclose(to_f64(delta), ref_delta, rtol=1e-5, atol=1e-5)


def test_bwd_head_dim_96_chained_long(cuda_device):
    """fwd → bwd at D = 96, S = 4096, sampled rows of two heads."""
    shape = (1, 4, 4096, 96)
    q, k, v = make_qkv(shape, seed=150)
    dout = _dout(shape, 151)
    scale = default_scale(96)
    out, lse = run_gpu(q, k, v, scale, True)
    dev = [x.to("cuda:0") for x in (q, k, v, out, lse, dout)]
    dq, dk, dv, _ = binding.attn_bwd(*dev, scale=scale, causal=True)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    n = [x.float().numpy() for x in (q, k, v, dout)]
    rng = np.random.default_rng(152)
    rows = np.unique(np.concatenate([[0, 127, 128, 4095], rng.integers(0, 4096, 120)]))
    for h in (0, 3):
        rq, rk, rv = attention_bwd_rows(*n, scale, True, 0, h, rows, rows)
        Mq, Mk, Mv = bwd_magnitudes(*n, scale, True, 0, h, rows, rows)
        compare_grad(to_f64(dq.cpu())[0, h, rows], rq, Mq, f"D=96 dq h{h}")
        compare_grad(to_f64(dk.cpu())[0, h, rows], rk, Mk, f"D=96 dk h{h}")
        compare_grad(to_f64(dv.cpu())[0, h, rows], rv, Mv, f"D=96 dv h{h}")


def test_head_dim_rules_on_gpu(cuda_device):
    """D not a multiple of 8 or above 256: refused before any launch, outputs
    untouched."""
    for D in (100, 264):
        q, k, v = (x.to("cuda:0") for x in make_qkv((1, 1, 64, D), seed=160))
        out = torch.full_like(q, SENTINEL)
        lse = torch.full((1, 1, 64), SENTINEL, device="cuda:0")
        if D % 8 or D > 256:
            with pytest.raises(binding.AttnError) as e:
                binding.attn_fwd(q, k, v, out=out, lse=lse)
            assert e.value.code == binding.ATTN_ERR_UNSUPPORTED
            torch.cuda.synchronize()
            assert (out == SENTINEL).all() and (lse == SENTINEL).all()

