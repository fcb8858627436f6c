"""GPU parity of the backward (attn_bwd) against the fp64 gradient oracle.

Every call goes through the C ABI.  The oracle sees only q, k, v and dout; the
kernel additionally gets out and lse, here from the oracle's forward (out
rounded to bf16, lse to fp32) so that the backward is tested on its own, and
in one test from the CUDA forward as a user would chain them.  Bar: the
element-wise bound of ``gpu_helpers.compare_grad`` (derived there from the
rounding steps of the kernel) and a relative Frobenius error <= 2^-7.
"""
import numpy as np
import pytest
import torch

from exact_attention_68_gb300 import binding
from exact_attention_68_gb300.workloads import WORKLOADS, default_scale, make_qkv
from gpu_helpers import bwd_magnitudes, compare_grad, run_gpu, to_f64
from oracle import attention_bwd, attention_bwd_rows, attention_fwd

pytestmark = pytest.mark.gpu


def _dout(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _oracle_out_lse(q, k, v, scale, causal):
    out, lse = attention_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), scale, causal)
    return (torch.from_numpy(out).to(torch.bfloat16), torch.from_numpy(lse).to(torch.float32))


def _run_bwd(q, k, v, out, lse, dout, scale, causal, device="cuda:0"):
    args = [x.to(device) for x in (q, k, v, out, lse, dout)]
    dq, dk, dv, delta = binding.attn_bwd(*args, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    return dq.cpu(), dk.cpu(), dv.cpu(), delta.cpu()


def _check_full(q, k, v, dout, dq, dk, dv, scale, causal, what):
    n = [x.float().numpy() for x in (q, k, v, dout)]
    rq, rk, rv = attention_bwd(*n, scale, causal)
    B, H, S, _ = q.shape
    rows = np.arange(S)
    res = {}
    for b in range(B):
        for h in range(H):
            Mq, Mk, Mv = bwd_magnitudes(*n, scale, causal, b, h, rows, rows)
            res[(b, h)] = (
                compare_grad(to_f64(dq)[b, h], rq[b, h], Mq, f"{what} dq b{b}h{h}"),
                compare_grad(to_f64(dk)[b, h], rk[b, h], Mk, f"{what} dk b{b}h{h}"),
                compare_grad(to_f64(dv)[b, h], rv[b, h], Mv, f"{what} dv b{b}h{h}"),
            )
    return res


SHAPES = [(1, 1, 1, 64), (1, 1, 7, 128), (1, 2, 128, 64), (2, 3, 129, 64), (1, 2, 200, 128),
          (1, 1, 256, 128), (1, 2, 384, 64), (2, 1, 513, 128), (3, 1, 1000, 64)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_bwd_full_oracle(cuda_device, shape, causal):
    q, k, v = make_qkv(shape, seed=41)
    dout = _dout(shape, 42)
    scale = default_scale(shape[3])
    out, lse = _oracle_out_lse(q, k, v, scale, causal)
    dq, dk, dv, delta = _run_bwd(q, k, v, out, lse, dout, scale, causal)
    _check_full(q, k, v, dout, dq, dk, dv, scale, causal, f"{shape} causal={causal}")
    # delta is rowsum(dout ⊙ out) of the bf16 out the kernel was given (fp32 sum)
    ref_delta = (dout.double() * out.double()).sum(-1).numpy()
    np.testing.assert_allclose(to_f64(delta), ref_delta, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("scale,qk_std", [(0.03, 1.0), (0.5, 2.0)])
def test_bwd_other_scales_and_peaked_softmax(cuda_device, scale, qk_std):
    shape = (2, 2, 300, 128)
    q, k, v = make_qkv(shape, seed=43, qk_std=qk_std)
    dout = _dout(shape, 44)
    for causal in (True, False):
        out, lse = _oracle_out_lse(q, k, v, scale, causal)
        dq, dk, dv, _ = _run_bwd(q, k, v, out, lse, dout, scale, causal)
        _check_full(q, k, v, dout, dq, dk, dv, scale, causal, f"scale={scale} causal={causal}")


def test_bwd_chained_with_cuda_forward(cuda_device):
    """fwd → bwd on the GPU as a user chains them (out, lse from attn_fwd)."""
    shape = (2, 4, 1024, 128)
    q, k, v = make_qkv(shape, seed=45)
    dout = _dout(shape, 46)
    scale = default_scale(128)
    out, lse = run_gpu(q, k, v, scale, True)
    dq, dk, dv, _ = _run_bwd(q, k, v, out, lse, dout, scale, True)
    _check_full(q, k, v, dout, dq, dk, dv, scale, True, "chained")


@pytest.mark.parametrize("name", ["c3", "c5"])
def test_bwd_workload_sampled_rows(cuda_device, name):
    """Full-size workloads: every row of two heads' dq, dk, dv (c3) or 384
    sampled rows of each of two heads (c5), against the oracle's row form."""
    w = WORKLOADS[name]
    q, k, v = make_qkv(w, seed=0)
    dout = _dout(w.shape, 47)
    scale = default_scale(w.D)
    # out and lse from the CUDA forward (running the fp64 forward over every
    # head is out of reach here); the oracle below recomputes its own
    out, lse = run_gpu(q, k, v, scale, w.causal)
    dq, dk, dv, _ = _run_bwd(q, k, v, out, lse, dout, scale, w.causal)
    n = [x.float().numpy() for x in (q, k, v, dout)]
    rng = np.random.default_rng(48)
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    for b, h in heads:
        if name == "c3":
            rows = np.arange(w.S)
        else:
            rows = np.unique(np.concatenate([[0, 1, 127, 128, w.S - 129, w.S - 1],
                                             rng.integers(0, w.S, 378)]))
        rq, rk, rv = attention_bwd_rows(*n, scale, w.causal, b, h, rows, rows)
        Mq, Mk, Mv = bwd_magnitudes(*n, scale, w.causal, b, h, rows, rows)
        compare_grad(to_f64(dq)[b, h, rows], rq, Mq, f"{name} dq b{b}h{h}")
        compare_grad(to_f64(dk)[b, h, rows], rk, Mk, f"{name} dk b{b}h{h}")
        compare_grad(to_f64(dv)[b, h, rows], rv, Mv, f"{name} dv b{b}h{h}")
    # every head: finite, and dv sums to the dout sum over the sequence
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    dv_sum = to_f64(dv).sum(axis=2)
    do_sum = to_f64(dout).sum(axis=2)
    assert np.abs(dv_sum - do_sum).max() <= 2.0 ** -6 * np.abs(to_f64(dout)).sum(axis=2).max()


def test_bwd_bitwise_deterministic(cuda_device):
    shape = (2, 4, 700, 128)
    q, k, v = make_qkv(shape, seed=49)
    dout = _dout(shape, 50)
    scale = default_scale(128)
    out, lse = _oracle_out_lse(q, k, v, scale, True)
    a = _run_bwd(q, k, v, out, lse, dout, scale, True)
    b = _run_bwd(q, k, v, out, lse, dout, scale, True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_bwd_causal_grads_of_last_key_come_from_last_query_only(cuda_device):
    """Causal: key S-1 is seen by query S-1 alone, so dk, dv of the last key
    depend on that query's row only (change every other dout row: unchanged)."""
    shape = (1, 2, 257, 64)
    q, k, v = make_qkv(shape, seed=51)
    scale = default_scale(64)
    out, lse = _oracle_out_lse(q, k, v, scale, True)
    d1 = _dout(shape, 52)
    d2 = d1.clone()
    d2[:, :, :-1] = _dout((1, 2, 256, 64), 53)
    _, dk1, dv1, _ = _run_bwd(q, k, v, out, lse, d1, scale, True)
    _, dk2, dv2, _ = _run_bwd(q, k, v, out, lse, d2, scale, True)
    assert torch.equal(dk1[:, :, -1], dk2[:, :, -1]) and torch.equal(dv1[:, :, -1], dv2[:, :, -1])


def test_bwd_long_context_32768(cuda_device):
    """S = 32768, one head: 256 K/V tiles per dq CTA and 256 Q tiles per dk/dv
    CTA; 160 sampled rows of dq, dk, dv against the oracle's row form."""
    shape = (1, 1, 32768, 128)
    q, k, v = make_qkv(shape, seed=71)
    dout = _dout(shape, 72)
    scale = default_scale(128)
    out, lse = run_gpu(q, k, v, scale, True)
    dq, dk, dv, _ = _run_bwd(q, k, v, out, lse, dout, scale, True)
    n = [x.float().numpy() for x in (q, k, v, dout)]
    rng = np.random.default_rng(73)
    rows = np.unique(np.concatenate([[0, 127, 128, 32767 - 128, 32767], rng.integers(0, 32768, 155)]))
    rq, rk, rv = attention_bwd_rows(*n, scale, True, 0, 0, rows, rows)
    Mq, Mk, Mv = bwd_magnitudes(*n, scale, True, 0, 0, rows, rows)
    compare_grad(to_f64(dq)[0, 0, rows], rq, Mq, "S=32768 dq")
    compare_grad(to_f64(dk)[0, 0, rows], rk, Mk, "S=32768 dk")
    compare_grad(to_f64(dv)[0, 0, rows], rv, Mv, "S=32768 dv")
