"""ctypes binding to the C ABI of include/attn.h (argument marshalling only).

Every step of the forward runs in the CUDA library; this module checks
dtypes/shapes, hands raw device pointers and the current CUDA stream to the C
functions and turns status codes into exceptions.  torch is used only to own
device memory and to name the stream.  If the library has not been built the
first call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from .build import LIB_PATH

__all__ = ["AttnError", "load_library", "attn_fwd", "attn_fwd_bounded", "attn_fwd_staged",
           "attn_fwd_noalloc", "attn_bwd", "attn_bwd_bounded", "attention", "device_status",
           "shard_range", "attn_fwd_sharded",
           "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_MISALIGNED",
           "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT", "ATTN_ERR_DEVICE_CHECK", "ATTN_BF16", "ATTN_F16", "EXPORTED_SYMBOLS"]

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED = 0, 1, 2
ATTN_ERR_MISALIGNED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = 3, 4, 5
ATTN_ERR_DEVICE_CHECK = 6
ATTN_BF16, ATTN_F16 = 0, 1
ATTN_DEFAULT_WAIT_TIMEOUT_NS = 2_000_000_000

_i64, _p, _f, _i, _u64 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int, ctypes.c_uint64
_SIGS = {
    "attn_fwd": (_i, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _f, _i, _p]),
    "attn_fwd_staged": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                             _i64, _i64, _i64, _i64, _f, _i, _p]),
    "attn_fwd_bounded": (_i, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _f, _i, _u64, _p]),
    "attn_fwd_noalloc": (_i, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _f, _i, _i, _p]),
    "attn_bwd": (_i, [_p] * 10 + [_i64, _i64, _i64, _i64, _f, _i, _p]),
    "attn_bwd_bounded": (_i, [_p] * 10 + [_i64, _i64, _i64, _i64, _f, _i, _u64, _p]),
    "attn_fwd_ex": (_i, [_p] * 5 + [_i64, _i64, _i64, _i64, _f, _i, _i, _u64, _p]),
    "attn_bwd_ex": (_i, [_p] * 10 + [_i64, _i64, _i64, _i64, _f, _i, _i, _u64, _p]),
    "attn_device_status": (_i, [_p]),
    "attn_status_string": (ctypes.c_char_p, [_i]),
    "attn_abi_version": (_i, []),
    "attn_last_cuda_error": (_i, []),
    "attn_shard_range": (_i, [_i64, _i, _i, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]),
}
EXPORTED_SYMBOLS = tuple(_SIGS)

_lib = None
_lock = threading.Lock()


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = _status_string(code)
        if code == ATTN_ERR_CUDA:
            msg += f" ({_cuda_cause()})"
        super().__init__(f"{where}: {msg} (status {code})")


def _cuda_cause() -> str:
    """The library's record of the CUDA failure behind the last ATTN_ERR_CUDA."""
    try:
        c = int(load_library().attn_last_cuda_error())
    except Exception:
        return "cause unknown"
    if c == -1:
        return "TMA tensor map encode failed"
    try:
        from cuda.bindings import runtime as _rt
        return f"{_rt.cudaError_t(c).name} ({c})"
    except Exception:
        return f"cudaError_t {c}"


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load (once) the CUDA library and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library not built: {p} is missing "
                               "(run `python -m exact_attention_68_gb300.build`)")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def _status_string(code: int) -> str:
    try:
        return load_library().attn_status_string(int(code)).decode()
    except Exception:  # library missing: still report the number
        return "attention library status"


def _stream_handle(device: torch.device, stream) -> int:
    s = torch.cuda.current_stream(device) if stream is None else stream
    return int(s.cuda_stream)


_DTYPES = {torch.bfloat16: ATTN_BF16, torch.float16: ATTN_F16}


def _check_qkv(q, k, v, allow_f16=False):
    """Checks q, k, v; returns the library's dtype code for them."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16 and not (allow_f16 and t.dtype == torch.float16):
            raise TypeError(f"{name} must be bfloat16" + (" or float16" if allow_f16 else ""))
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, S, D] tensor")
    if not (q.shape == k.shape == v.shape) or not (q.device == k.device == v.device):
        raise ValueError("q, k, v must share shape and device")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    return _DTYPES[q.dtype]


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
             causal: bool = True, out: torch.Tensor | None = None,
             lse: torch.Tensor | None = None, stream=None):
    """Fused attention forward.  Returns (out bf16 [B,H,S,D], lse fp32 [B,H,S])."""
    return attn_fwd_bounded(q, k, v, scale, causal, out, lse, stream, None)


def attn_fwd_bounded(q, k, v, scale=None, causal=True, out=None, lse=None, stream=None,
                     wait_timeout_ns: int | None = None):
    """attn_fwd with an explicit bound on every in-kernel wait (None = library default).
    q, k, v may be bfloat16 or float16; out has their dtype."""
    dt = _check_qkv(q, k, v, allow_f16=True)
    B, H, S, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    if (out.dtype != q.dtype or out.shape != q.shape or not out.is_contiguous()
            or out.device != q.device):
        raise ValueError("out must be a contiguous tensor shaped like q, of its dtype and device")
    if (lse.dtype != torch.float32 or lse.shape != (B, H, S) or not lse.is_contiguous()
            or lse.device != q.device):
        raise ValueError("lse must be a contiguous fp32 [B, H, S] tensor on q's device")
    lib = load_library()
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
            B, H, S, D, float(scale), 1 if causal else 0)
    with torch.cuda.device(q.device):
        st = _stream_handle(q.device, stream)
        if dt == ATTN_F16:
            tmo = ATTN_DEFAULT_WAIT_TIMEOUT_NS if wait_timeout_ns is None else int(wait_timeout_ns)
            rc = lib.attn_fwd_ex(*args, dt, tmo, st)
        elif wait_timeout_ns is None:
            rc = lib.attn_fwd(*args, st)
        else:
            rc = lib.attn_fwd_bounded(*args, int(wait_timeout_ns), st)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return out, lse


def attn_fwd_staged(q_h, k_h, v_h, out_h, lse_h, q_d, k_d, v_d, out_d, lse_d, scale=None,
                    causal=True, stream=None):
    """Forward from host buffers: H2D copies, kernel, D2H copies on one stream."""
    _check_qkv(q_d, k_d, v_d)
    B, H, S, D = q_d.shape
    for name, t in (("q_h", q_h), ("k_h", k_h), ("v_h", v_h), ("out_h", out_h), ("lse_h", lse_h)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    # the library copies whole [B, H, S, D] bf16 (and [B, H, S] fp32) buffers
    # between these tensors: every one must have exactly that size and type
    for name, t in (("q_h", q_h), ("k_h", k_h), ("v_h", v_h), ("out_h", out_h)):
        if t.dtype != torch.bfloat16 or t.shape != q_d.shape:
            raise ValueError(f"{name} must be a bf16 tensor shaped like q_d")
    if lse_h.dtype != torch.float32 or lse_h.shape != (B, H, S):
        raise ValueError("lse_h must be an fp32 [B, H, S] tensor")
    if (not isinstance(out_d, torch.Tensor) or out_d.dtype != torch.bfloat16
            or out_d.shape != q_d.shape or not out_d.is_contiguous() or out_d.device != q_d.device):
        raise ValueError("out_d must be a contiguous bf16 tensor shaped like q_d, on its device")
    if (not isinstance(lse_d, torch.Tensor) or lse_d.dtype != torch.float32
            or lse_d.shape != (B, H, S) or not lse_d.is_contiguous() or lse_d.device != q_d.device):
        raise ValueError("lse_d must be a contiguous fp32 [B, H, S] tensor on q_d's device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lib = load_library()
    with torch.cuda.device(q_d.device):
        rc = lib.attn_fwd_staged(q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(), out_h.data_ptr(),
                                 lse_h.data_ptr(), q_d.data_ptr(), k_d.data_ptr(), v_d.data_ptr(),
                                 out_d.data_ptr(), lse_d.data_ptr(), B, H, S, D, float(scale),
                                 1 if causal else 0, _stream_handle(q_d.device, stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_staged")
    return out_h, lse_h


def attn_fwd_noalloc(q, k, v, out, lse, scale=None, causal=True, check_status=True, stream=None):
    """Forward through attn_fwd_noalloc: the library allocates no device memory.

    ``out`` and ``lse`` are required (the caller owns all memory).  With
    ``check_status`` the call synchronises the stream and raises AttnError if
    the kernel recorded an in-kernel wait that ran out.
    """
    _check_qkv(q, k, v)
    B, H, S, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if (out.dtype != torch.bfloat16 or out.shape != q.shape or not out.is_contiguous()
            or out.device != q.device):
        raise ValueError("out must be a contiguous bf16 tensor shaped like q, on its device")
    if (lse.dtype != torch.float32 or lse.shape != (B, H, S) or not lse.is_contiguous()
            or lse.device != q.device):
        raise ValueError("lse must be a contiguous fp32 [B, H, S] tensor on q's device")
    lib = load_library()
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr(), B, H, S, D, float(scale), 1 if causal else 0,
                                  1 if check_status else 0, _stream_handle(q.device, stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_noalloc")
    return out, lse


def attn_bwd(q, k, v, out, lse, dout, scale=None, causal=True, dq=None, dk=None, dv=None,
             delta=None, stream=None):
    """Gradient of attn_fwd.  Returns (dq, dk, dv) bf16 [B,H,S,D] and delta fp32 [B,H,S]."""
    return attn_bwd_bounded(q, k, v, out, lse, dout, scale, causal, dq, dk, dv, delta, stream, None)


def attn_bwd_bounded(q, k, v, out, lse, dout, scale=None, causal=True, dq=None, dk=None, dv=None,
                     delta=None, stream=None, wait_timeout_ns: int | None = None):
    """attn_bwd with an explicit bound on every in-kernel wait (None = library default).
    The 16-bit tensors may be bfloat16 or float16 (all the same)."""
    dt = _check_qkv(q, k, v, allow_f16=True)
    B, H, S, D = q.shape
    for name, t in (("out", out), ("dout", dout)):
        if (not isinstance(t, torch.Tensor) or t.dtype != q.dtype or t.shape != q.shape
                or not t.is_contiguous() or t.device != q.device):
            raise ValueError(f"{name} must be a contiguous tensor shaped like q, of its dtype and device")
    if (not isinstance(lse, torch.Tensor) or lse.dtype != torch.float32 or lse.shape != (B, H, S)
            or not lse.is_contiguous() or lse.device != q.device):
        raise ValueError("lse must be a contiguous fp32 [B, H, S] tensor on q's device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    delta = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if delta is None else delta
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        if (t.dtype != q.dtype or t.shape != q.shape or not t.is_contiguous()
                or t.device != q.device):
            raise ValueError(f"{name} must be a contiguous tensor shaped like q, of its dtype and device")
    if (delta.dtype != torch.float32 or delta.shape != (B, H, S) or not delta.is_contiguous()
            or delta.device != q.device):
        raise ValueError("delta must be a contiguous fp32 [B, H, S] tensor on q's device")
    lib = load_library()
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
            dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), delta.data_ptr(),
            B, H, S, D, float(scale), 1 if causal else 0)
    with torch.cuda.device(q.device):
        st = _stream_handle(q.device, stream)
        if dt == ATTN_F16:
            tmo = ATTN_DEFAULT_WAIT_TIMEOUT_NS if wait_timeout_ns is None else int(wait_timeout_ns)
            rc = lib.attn_bwd_ex(*args, dt, tmo, st)
        elif wait_timeout_ns is None:
            rc = lib.attn_bwd(*args, st)
        else:
            rc = lib.attn_bwd_bounded(*args, int(wait_timeout_ns), st)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")
    return dq, dk, dv, delta


def device_status(device=None, stream=None) -> int:
    """Synchronise the stream, read and clear the device status word (0 = ok)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    lib = load_library()
    with torch.cuda.device(dev):
        return int(lib.attn_device_status(_stream_handle(dev, stream)))


def shard_range(units: int, world: int, rank: int):
    """(first, count): the contiguous range of the `units` (b, h) slices that
    rank `rank` of `world` takes (attn_shard_range of the C ABI)."""
    first, count = ctypes.c_int64(0), ctypes.c_int64(0)
    rc = load_library().attn_shard_range(int(units), int(world), int(rank), ctypes.byref(first),
                                         ctypes.byref(count))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_shard_range")
    return first.value, count.value


def attn_fwd_sharded(q, k, v, scale=None, causal=True, rank=None, world=None, device=None,
                     stream=None):
    """This rank's share of one forward split over processes, one per GPU.

    q, k, v: the whole problem's contiguous [B, H, S, D] bf16/fp16 tensors, on
    the host or on this rank's GPU.  rank / world default to the
    torch.distributed process group's.  The rank takes the slices
    shard_range(B·H, world, rank) gives it, moves only those to `device`
    (default: the current CUDA device) and runs attn_fwd on them as one
    [1, count, S, D] problem.  Nothing is exchanged between ranks.  Returns
    (first, count, out [count, S, D], lse [count, S]) on `device`; count may be
    0 (then out and lse are empty).
    """
    if rank is None or world is None:
        import torch.distributed as dist
        rank = dist.get_rank() if rank is None else rank
        world = dist.get_world_size() if world is None else world
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, S, D] tensor")
    if not (q.shape == k.shape == v.shape):
        raise ValueError("q, k, v must share a shape")
    B, H, S, D = q.shape
    first, count = shard_range(B * H, world, rank)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if count == 0:
        return first, 0, torch.empty((0, S, D), dtype=q.dtype, device=dev), \
            torch.empty((0, S), dtype=torch.float32, device=dev)
    part = [t.view(B * H, S, D)[first:first + count].to(dev).unsqueeze(0) for t in (q, k, v)]
    out, lse = attn_fwd(*part, scale=scale, causal=causal, stream=stream)
    return first, count, out[0], lse[0]


class _AttentionFn(torch.autograd.Function):
    """attn_fwd in forward, attn_bwd in backward (both through the C ABI)."""

    @staticmethod
    def forward(ctx, q, k, v, scale, causal):
        out, lse = attn_fwd(q, k, v, scale=scale, causal=causal)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.scale, ctx.causal = scale, causal
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse = ctx.saved_tensors
        dq, dk, dv, _ = attn_bwd(q, k, v, out, lse, dout.contiguous(), scale=ctx.scale,
                                 causal=ctx.causal)
        return dq, dk, dv, None, None


def attention(q, k, v, scale=None, causal=True):
    """Differentiable fused attention: out = softmax(scale·q·kᵀ + mask)·v for
    contiguous bf16/fp16 CUDA tensors [B, H, S, D]; gradients flow to q, k, v."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return _AttentionFn.apply(q, k, v, float(scale), bool(causal))
