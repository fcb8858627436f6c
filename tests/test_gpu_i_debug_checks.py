"""The debug build (-DATTN_DEBUG) on the GPU: every kernel checks the index
arithmetic of each memory access before making it (TMA coordinates and
column alignment, shared- and tensor-memory addresses against the CTA's
allocation, rows and columns of plain global accesses) and reports a failed
check as ATTN_ERR_DEVICE_CHECK instead of making the access.  Here the debug
kernels run over ragged shapes, every kernel width, padded head dimensions,
both masks and both 16-bit types: no check may fail, and the results must
still meet the oracle's bars."""
import numpy as np
import pytest
import torch

from exact_attention_68_gb300 import binding
from exact_attention_68_gb300.build import build_debug_library
from exact_attention_68_gb300.workloads import default_scale, make_qkv
from gpu_helpers import bwd_magnitudes, compare, compare_grad, to_f64
from oracle import attention_bwd, attention_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg(cuda_device):
    return binding.load_library(build_debug_library())


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _fwd(lib, q, k, v, scale, causal):
    B, H, S, D = q.shape
    qd, kd, vd = (x.to("cuda:0") for x in (q, k, v))
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda:0")
    dt = binding.ATTN_F16 if q.dtype == torch.float16 else binding.ATTN_BF16
    rc = lib.attn_fwd_ex(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), lse.data_ptr(),
                         B, H, S, D, scale, int(causal), dt, binding.ATTN_DEFAULT_WAIT_TIMEOUT_NS,
                         _stream())
    assert rc == binding.ATTN_OK
    assert lib.attn_device_status(_stream()) == binding.ATTN_OK
    return out.cpu(), lse.cpu()


FWD_CASES = [(64, (1, 2, 1)), (64, (2, 1, 300)), (128, (1, 2, 129)), (128, (2, 2, 1000)),
             (256, (1, 2, 65)), (256, (1, 1, 513)), (32, (1, 2, 200)), (96, (2, 1, 257)),
             (192, (1, 2, 130)), (136, (2, 1, 200)), (8, (1, 1, 77)),
             # long enough that the persistent kernel takes the path whose
             # softmax warps load Q (more than 24 K/V steps a tile on average
             # under both masks), ragged in S
             (128, (1, 1, 6500)), (64, (1, 1, 6500))]


@pytest.mark.parametrize("D,bhs", FWD_CASES, ids=lambda x: str(x))
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
def test_debug_forward_no_check_fails(dbg, D, bhs, causal, dtype):
    shape = (*bhs, D)
    q, k, v = make_qkv(shape, seed=170 + D, dtype=dtype)
    scale = default_scale(D)
    out, lse = _fwd(dbg, q, k, v, scale, causal)
    ro, rl = attention_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale, causal)
    compare(to_f64(out), to_f64(lse), ro, rl, f"debug D={D} {shape} causal={causal} {dtype}")


@pytest.mark.parametrize("D,bhs", [(64, (1, 2, 1)), (64, (2, 1, 300)), (128, (1, 2, 129)),
                                   (128, (1, 1, 513)), (40, (1, 2, 200)), (96, (2, 1, 257)),
                                   (256, (1, 2, 129)), (136, (2, 1, 200))],
                         ids=lambda x: str(x))
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_debug_backward_no_check_fails(dbg, D, bhs, causal):
    shape = (*bhs, D)
    q, k, v = make_qkv(shape, seed=180 + D)
    g = torch.Generator().manual_seed(181 + D)
    dout = torch.randn(shape, generator=g).to(torch.bfloat16)
    scale = default_scale(D)
    n = [x.double().numpy() for x in (q, k, v, dout)]
    ro, rl = attention_fwd(*n[:3], scale, causal)
    out = torch.from_numpy(ro).to(torch.bfloat16)
    lse = torch.from_numpy(rl).float()
    dev = [x.to("cuda:0") for x in (q, k, v, out, lse, dout)]
    dq, dk, dv = (torch.empty_like(dev[0]) for _ in range(3))
    delta = torch.empty(shape[:3], dtype=torch.float32, device="cuda:0")
    B, H, S, _ = shape
    rc = dbg.attn_bwd(*(t.data_ptr() for t in dev), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                      delta.data_ptr(), B, H, S, D, scale, int(causal), _stream())
    assert rc == binding.ATTN_OK
    assert dbg.attn_device_status(_stream()) == binding.ATTN_OK
    rq, rk, rv = attention_bwd(*n, scale, causal)
    rows = np.arange(S)
    for b in range(B):
        for h in range(H):
            Mq, Mk, Mv = bwd_magnitudes(*n, scale, causal, b, h, rows, rows)
            compare_grad(to_f64(dq.cpu())[b, h], rq[b, h], Mq, f"debug D={D} dq")
            compare_grad(to_f64(dk.cpu())[b, h], rk[b, h], Mk, f"debug D={D} dk")
            compare_grad(to_f64(dv.cpu())[b, h], rv[b, h], Mv, f"debug D={D} dv")


def test_debug_staged_and_noalloc_entry_points(dbg):
    shape = (2, 3, 300, 128)
    q, k, v = make_qkv(shape, seed=190)
    scale = default_scale(128)
    B, H, S, D = shape
    q_h, k_h, v_h = (x.pin_memory() for x in (q, k, v))
    out_h = torch.empty_like(q_h).pin_memory()
    lse_h = torch.empty((B, H, S), dtype=torch.float32).pin_memory()
    q_d, k_d, v_d = (torch.empty_like(x, device="cuda:0") for x in (q, k, v))
    out_d = torch.empty_like(q_d)
    lse_d = torch.empty((B, H, S), dtype=torch.float32, device="cuda:0")
    rc = dbg.attn_fwd_staged(q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(), out_h.data_ptr(),
                             lse_h.data_ptr(), q_d.data_ptr(), k_d.data_ptr(), v_d.data_ptr(),
                             out_d.data_ptr(), lse_d.data_ptr(), B, H, S, D, scale, 1, _stream())
    assert rc == binding.ATTN_OK
    assert dbg.attn_device_status(_stream()) == binding.ATTN_OK
    ro, rl = attention_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale, True)
    compare(to_f64(out_h), to_f64(lse_h), ro, rl, "debug staged")
    out2 = torch.empty_like(q_d)
    lse2 = torch.empty_like(lse_d)
    rc = dbg.attn_fwd_noalloc(q_d.data_ptr(), k_d.data_ptr(), v_d.data_ptr(), out2.data_ptr(),
                              lse2.data_ptr(), B, H, S, D, scale, 1, 1, _stream())
    assert rc == binding.ATTN_OK
    assert torch.equal(out2.cpu(), out_h) and torch.equal(lse2.cpu(), lse_h)
