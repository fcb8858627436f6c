"""GPU unit test of the tcgen05 operand conventions (descriptors, TMEM packing).

Small-integer inputs make every product and sum exact in fp32, so the tensor
core result must equal the CPU matmul bit for bit.  A wrong swizzle, stride,
major-ness, N/M field or bf16 packing order shows up as a mismatch.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_attention_68_gb300.build import build_unit_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def unit_lib(cuda_device):
    lib = ctypes.CDLL(build_unit_library())
    lib.umma_unit_run.restype = ctypes.c_int
    lib.umma_unit_run.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int, ctypes.c_int]
    return lib


@pytest.mark.parametrize("predicated", [0, 1], ids=["lane0", "predicated"])
@pytest.mark.parametrize("D", [64, 128])
def test_qk_and_pv_mma_are_exact(unit_lib, D, predicated):
    # predicated: the whole MMA warp runs the issue path with each product and
    # commit predicated on lane 0 (the backward kernels' form); a product
    # issued by more than one lane would accumulate more than once
    g = torch.Generator().manual_seed(D)
    a = torch.randint(-2, 3, (128, D), generator=g).to(torch.bfloat16)
    b = torch.randint(-2, 3, (128, D), generator=g).to(torch.bfloat16)
    v = torch.randint(-3, 4, (128, D), generator=g).to(torch.bfloat16)
    p = torch.randint(-2, 3, (128, 128), generator=g).to(torch.bfloat16)
    # make the two halves of each packed pair distinguishable
    p[:, 1::2] *= 2
    packed = p.view(torch.int16).to(torch.int32) & 0xFFFF
    packed = (packed[:, 0::2] | (packed[:, 1::2] << 16)).to(torch.int32).contiguous()
    dev = "cuda:0"
    ad, bd, vd, pd = (x.contiguous().to(dev) for x in (a, b, v, packed))
    s_out = torch.full((128, 128), float("nan"), device=dev)
    o_out = torch.full((128, D), float("nan"), device=dev)
    status = torch.zeros(2, dtype=torch.int32, device=dev)
    rc = unit_lib.umma_unit_run(ad.data_ptr(), bd.data_ptr(), vd.data_ptr(), pd.data_ptr(),
                                s_out.data_ptr(), o_out.data_ptr(), status.data_ptr(), D, predicated)
    assert rc == 0
    assert status.cpu().tolist() == [0, 0]
    s_ref = a.double().numpy() @ b.double().numpy().T
    o_ref = p.double().numpy() @ v.double().numpy()
    np.testing.assert_array_equal(s_out.cpu().double().numpy(), s_ref)
    np.testing.assert_array_equal(o_out.cpu().double().numpy(), o_ref)
