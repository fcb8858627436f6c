"""CPU checks of the C-ABI library: it loads, exports every declared symbol,
and rejects bad arguments before touching the GPU (no compute call here)."""
import ctypes
import os
import re

import pytest

from exact_attention_68_gb300 import binding
from exact_attention_68_gb300.build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    path = build_library()
    return binding.load_library(path)


def _declared():
    with open(HEADER) as f:
        src = f.read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", src)


def test_header_declares_the_bound_symbols():
    names = _declared()
    assert sorted(names) == sorted(binding.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert lib.attn_abi_version() == 1


def test_status_strings(lib):
    for code in range(7):
        assert lib.attn_status_string(code) != b"unknown status"
    assert lib.attn_status_string(0) == b"ok"
    assert b"debug" in lib.attn_status_string(binding.ATTN_ERR_DEVICE_CHECK)


def test_debug_build_compiles_and_exports_the_abi():
    """The -DATTN_DEBUG variant (in-kernel index checks) builds for sm_103a
    and exports the same C ABI; its kernels run in the GPU tests."""
    from exact_attention_68_gb300.build import build_debug_library
    path = build_debug_library()
    dbg = binding.load_library(path)
    for name in binding.EXPORTED_SYMBOLS:
        assert hasattr(dbg, name), name
    assert dbg.attn_abi_version() == 1


# Fake, never dereferenced device addresses: validation runs before any CUDA call.
A = 0x7F0000000000
T = 1 << 30  # spacing large enough for the shapes used below


def _call(lib, q=A, k=A + T, v=A + 2 * T, out=A + 3 * T, lse=A + 4 * T,
          B=1, H=2, S=128, D=64, scale=0.125, causal=1):
    return lib.attn_fwd(q, k, v, out, lse, B, H, S, D, scale, causal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(k=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(v=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(out=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(lse=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(B=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(H=-1), binding.ATTN_ERR_INVALID_ARG),
    (dict(S=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(D=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(D=100), binding.ATTN_ERR_UNSUPPORTED),   # rows not a multiple of 16 bytes
    (dict(D=4), binding.ATTN_ERR_UNSUPPORTED),
    (dict(D=264), binding.ATTN_ERR_UNSUPPORTED),
    (dict(D=512), binding.ATTN_ERR_UNSUPPORTED),
    (dict(scale=0.0), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=-0.5), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), binding.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), binding.ATTN_ERR_INVALID_ARG),
    (dict(q=A + 8), binding.ATTN_ERR_MISALIGNED),
    (dict(out=A + 3 * T + 2), binding.ATTN_ERR_MISALIGNED),
    (dict(lse=A + 4 * T + 1), binding.ATTN_ERR_MISALIGNED),
    (dict(out=A), binding.ATTN_ERR_INVALID_ARG),                # out aliases q
    (dict(lse=A + 3 * T + 64), binding.ATTN_ERR_INVALID_ARG),   # lse inside out
    (dict(B=1 << 31), binding.ATTN_ERR_INVALID_ARG),
    (dict(B=1 << 20, H=1 << 20), binding.ATTN_ERR_INVALID_ARG),
    (dict(B=1 << 16, H=1 << 14, S=1 << 20), binding.ATTN_ERR_INVALID_ARG),
])
def test_invalid_arguments_are_rejected_before_launch(lib, kw, code):
    assert _call(lib, **kw) == code


def test_bounded_and_staged_validate_too(lib):
    assert lib.attn_fwd_bounded(0, A, A, A + 3 * T, A + 4 * T, 1, 1, 128, 64, 0.125, 1, 0, None) \
        == binding.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_staged(0, A, A, A, A, A, A + T, A + 2 * T, A + 3 * T, A + 4 * T,
                               1, 1, 128, 64, 0.125, 1, None) == binding.ATTN_ERR_INVALID_ARG
    # the same device buffer for q and k cannot hold two different host inputs
    assert lib.attn_fwd_staged(A, A, A, A, A, A, A, A + 2 * T, A + 3 * T, A + 4 * T,
                               1, 1, 128, 64, 0.125, 1, None) == binding.ATTN_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        binding.load_library(str(tmp_path / "missing.so"))


def test_noalloc_validates_before_touching_the_gpu(lib):
    args = [A, A + T, A + 2 * T, A + 3 * T, A + 4 * T, 1, 2, 128, 64, 0.125, 1]
    assert lib.attn_fwd_noalloc(*args, 2, None) == binding.ATTN_ERR_INVALID_ARG  # check_status
    bad = list(args)
    bad[0] = 0
    assert lib.attn_fwd_noalloc(*bad, 1, None) == binding.ATTN_ERR_INVALID_ARG
    bad = list(args)
    bad[8] = 84  # not a multiple of 8
    assert lib.attn_fwd_noalloc(*bad, 1, None) == binding.ATTN_ERR_UNSUPPORTED


def _bwd(lib, q=A, k=A + T, v=A + 2 * T, out=A + 3 * T, lse=A + 4 * T, dout=A + 5 * T,
         dq=A + 6 * T, dk=A + 7 * T, dv=A + 8 * T, delta=A + 9 * T,
         B=1, H=2, S=128, D=64, scale=0.125, causal=1):
    return lib.attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, delta, B, H, S, D, scale, causal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(out=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(lse=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(dout=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(dq=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(dk=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(dv=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(delta=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(S=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(D=100), binding.ATTN_ERR_UNSUPPORTED),
    (dict(D=264), binding.ATTN_ERR_UNSUPPORTED),   # above 256
    (dict(D=260), binding.ATTN_ERR_UNSUPPORTED),
    (dict(scale=0.0), binding.ATTN_ERR_INVALID_ARG),
    (dict(causal=3), binding.ATTN_ERR_INVALID_ARG),
    (dict(dout=A + 5 * T + 8), binding.ATTN_ERR_MISALIGNED),
    (dict(dq=A + 6 * T + 4), binding.ATTN_ERR_MISALIGNED),
    (dict(dv=A + 8 * T + 2), binding.ATTN_ERR_MISALIGNED),
    (dict(delta=A + 9 * T + 2), binding.ATTN_ERR_MISALIGNED),
    (dict(dq=A), binding.ATTN_ERR_INVALID_ARG),               # dq aliases q
    (dict(dk=A + 5 * T), binding.ATTN_ERR_INVALID_ARG),       # dk aliases dout
    (dict(dv=A + 6 * T + 64), binding.ATTN_ERR_INVALID_ARG),  # dv inside dq
    (dict(delta=A + 4 * T), binding.ATTN_ERR_INVALID_ARG),    # delta aliases lse
    (dict(delta=A + 8 * T + 128), binding.ATTN_ERR_INVALID_ARG),  # delta inside dv
])
def test_bwd_invalid_arguments_are_rejected_before_launch(lib, kw, code):
    assert _bwd(lib, **kw) == code


def test_bwd_bounded_validates_too(lib):
    args = [A, A + T, A + 2 * T, A + 3 * T, A + 4 * T, 0, A + 6 * T, A + 7 * T, A + 8 * T,
            A + 9 * T, 1, 2, 128, 64, 0.125, 1]
    assert lib.attn_bwd_bounded(*args, 0, None) == binding.ATTN_ERR_INVALID_ARG


def test_ex_entry_points_validate_dtype_first(lib):
    fwd = [A, A + T, A + 2 * T, A + 3 * T, A + 4 * T, 1, 2, 128, 64, 0.125, 1]
    assert lib.attn_fwd_ex(*fwd, 2, binding.ATTN_DEFAULT_WAIT_TIMEOUT_NS, None) == binding.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_ex(*fwd, -1, binding.ATTN_DEFAULT_WAIT_TIMEOUT_NS, None) == binding.ATTN_ERR_INVALID_ARG
    bad = list(fwd)
    bad[8] = 260
    assert lib.attn_fwd_ex(*bad, binding.ATTN_F16, 0, None) == binding.ATTN_ERR_UNSUPPORTED
    bwd = [A, A + T, A + 2 * T, A + 3 * T, A + 4 * T, A + 5 * T, A + 6 * T, A + 7 * T, A + 8 * T,
           A + 9 * T, 1, 2, 128, 64, 0.125, 1]
    assert lib.attn_bwd_ex(*bwd, 7, 0, None) == binding.ATTN_ERR_INVALID_ARG
    bad = list(bwd)
    bad[6] = A  # dq aliases q
    assert lib.attn_bwd_ex(*bad, binding.ATTN_F16, 0, None) == binding.ATTN_ERR_INVALID_ARG


def test_make_qkv_dtype():
    from exact_attention_68_gb300.workloads import make_qkv
    import torch
    qb = make_qkv((1, 1, 8, 64), seed=3)
    qh = make_qkv((1, 1, 8, 64), seed=3, dtype=torch.float16)
    assert all(t.dtype == torch.bfloat16 for t in qb) and all(t.dtype == torch.float16 for t in qh)
    # the same draws, rounded to the two types
    assert torch.allclose(qb[0].float(), qh[0].float(), atol=2e-2 * qh[0].abs().max().item())
