"""Shared helpers of the GPU parity tests (compare the CUDA path with the oracle)."""
import numpy as np
import torch

from exact_attention_68_gb300 import binding

# Tolerances on the bf16 output and the fp32 logsumexp, against the unrounded
# fp64 oracle: max |err| <= 2e-2, mean |err| <= 2e-3 (out), |err| <= 1e-3 (lse).
OUT_MAX_TOL = 2e-2
OUT_MEAN_TOL = 2e-3
LSE_TOL = 1e-3


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def run_gpu(q, k, v, scale, causal, device="cuda:0"):
    """Run the CUDA forward on CPU bf16 inputs; return (out, lse) on the CPU."""
    qd, kd, vd = (x.to(device) for x in (q, k, v))
    out, lse = binding.attn_fwd(qd, kd, vd, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    return out.cpu(), lse.cpu()


def compare(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    """Element-wise comparison; returns the error summary, asserts the bar."""
    og = np.asarray(out_gpu, np.float64)
    lg = np.asarray(lse_gpu, np.float64)
    assert np.isfinite(og).all(), f"{what}: non-finite output"
    assert np.isfinite(lg).all(), f"{what}: non-finite lse"
    err = np.abs(og - out_ref)
    lerr = np.abs(lg - lse_ref)
    summary = dict(out_max=float(err.max()), out_mean=float(err.mean()), lse_max=float(lerr.max()))
    assert summary["out_max"] <= OUT_MAX_TOL, (what, summary)
    assert summary["out_mean"] <= OUT_MEAN_TOL, (what, summary)
    assert summary["lse_max"] <= LSE_TOL, (what, summary)
    return summary
