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


# ---------------------------------------------------------------- backward
# Element-wise bar for the gradients.  The kernel rounds P and dS to bf16
# (unit roundoff 2^-8) before the tensor core multiplies them by exact bf16
# operands with fp32 accumulation, computes delta_i from the bf16 `out`
# (error <= 2^-8 · E_i, E_i = Σ_d |dout_id · out_id|) and rounds each gradient
# to bf16.  So each element obeys |err| <= 2^-8 · (M + |ref|) up to fp32
# terms, with M the magnitude sum of what it accumulates:
#   dv_j: Σ_i attn_ij |dout_i|
#   dk_j: scale · Σ_i (|dz_ij| + attn_ij E_i) |q_i|
#   dq_i: scale · Σ_j (|dz_ij| + attn_ij E_i) |k_j|
# The tests allow twice that, 2^-7, plus 1e-6 absolute.
BWD_REL = 2.0 ** -7
BWD_ABS = 1e-6


def bwd_magnitudes(q, k, v, dout, scale, causal, b, h, q_rows, kv_rows, chunk=1024):
    """M_q[q_rows], M_k[kv_rows], M_v[kv_rows] of one (b, h), float64 numpy."""
    qh, kh, vh, dh = (np.asarray(x[b, h], dtype=np.float64) for x in (q, k, v, dout))
    S = qh.shape[0]
    q_rows = np.asarray(q_rows, dtype=np.int64)
    kv_rows = np.asarray(kv_rows, dtype=np.int64)
    Mq = np.zeros((q_rows.size, qh.shape[1]))
    Mk = np.zeros((kv_rows.size, qh.shape[1]))
    Mv = np.zeros((kv_rows.size, qh.shape[1]))
    want_q = {int(r): n for n, r in enumerate(q_rows)}
    for r0 in range(0, S, chunk):
        rows = np.arange(r0, min(S, r0 + chunk))
        s = (qh[rows] @ kh.T) * scale
        if causal:
            s = np.where(np.arange(S)[None, :] > rows[:, None], -np.inf, s)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        attn = e / e.sum(axis=1, keepdims=True)
        out = attn @ vh
        dattn = dh[rows] @ vh.T
        delta = np.sum(dh[rows] * out, axis=1, keepdims=True)
        dz = np.abs(attn * (dattn - delta))
        E = np.sum(np.abs(dh[rows] * out), axis=1, keepdims=True)
        w = dz + attn * E                       # [rows, S]
        Mk += scale * (w[:, kv_rows].T @ np.abs(qh[rows]))
        Mv += attn[:, kv_rows].T @ np.abs(dh[rows])
        for n_local, r in enumerate(rows):
            if int(r) in want_q:
                Mq[want_q[int(r)]] = scale * (w[n_local] @ np.abs(kh))
    return Mq, Mk, Mv


def compare_grad(got, ref, mag, what=""):
    """Element-wise |got - ref| <= BWD_REL·(mag + |ref|) + BWD_ABS; returns a summary."""
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite gradient"
    err = np.abs(got - ref)
    bound = BWD_REL * (mag + np.abs(ref)) + BWD_ABS
    worst = float((err / bound).max()) if err.size else 0.0
    rel_fro = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30))
    summary = dict(worst_ratio=worst, max_err=float(err.max()) if err.size else 0.0,
                   rel_fro=rel_fro)
    assert worst <= 1.0, (what, summary)
    # the relative bar needs a reference to be relative to: a gradient that is
    # exactly zero (one key: its weight is 1 and dS = dP - delta = 0) is held
    # to the element-wise bound alone
    if np.linalg.norm(ref) > 0:
        assert rel_fro <= BWD_REL, (what, summary)
    return summary
