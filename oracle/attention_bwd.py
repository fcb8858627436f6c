"""Plain, slow, fp64 CPU oracle for the gradient of exact attention (backward).

TEST INFRASTRUCTURE. Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline / reference leg of ``bench.py`` may
import or run anything under ``oracle/``. The product path never calls it and
shares no code with it.

The pages define the forward only: the five steps of "Profiling in PyTorch
(Part 3): Attention is all you profile", section "Naive attention".  The same
page's passage on in-place operations notes that autograd's backward formulas
reuse values the forward saw.  The backward computed here is the exact
gradient of that forward with respect to q, k and v, for an upstream gradient
``dout`` = ∂L/∂out, taking the five steps in reverse with the chain rule:

  5. out  = attn · v             →  dattn = dout · vᵀ,   dv = attnᵀ · dout
  4. attn = softmax(z) per row   →  dz = attn ⊙ (dattn − rowsum(attn ⊙ dattn))
  3. z    = masked_fill(y, −inf) →  dy = dz (masked entries of attn are 0, so
                                       dz is 0 there already)
  2. y    = x · scale            →  dx = scale · dy
  1. x    = q · kᵀ               →  dq = dx · k,          dk = dxᵀ · q

rowsum(attn ⊙ dattn) equals dout_i · out_i for row i (substitute dattn =
dout · vᵀ and out = attn · v); ``attention_bwd`` uses the left form, the row
form below the right one.  A fully masked row (only possible without equal
query and key lengths) has attn = 0 and contributes nothing.
"""
from __future__ import annotations

import numpy as np

from .attention import _head_rows, _scores, causal_mask, softmax_rows

__all__ = ["attention_bwd", "attention_bwd_rows"]

_ROW_CHUNK = 1024


def _head_bwd(qh, kh, vh, douth, scale, causal):
    """The five steps in reverse for one (batch, head), full matrices."""
    S = qh.shape[0]
    rows = np.arange(S)
    attn, _ = softmax_rows(_scores(qh, kh, scale, causal, rows))   # forward steps 1-4
    dattn = douth @ vh.T                                             # step 5, w.r.t. attn
    dv = attn.T @ douth                                              # step 5, w.r.t. v
    dz = attn * (dattn - np.sum(attn * dattn, axis=1, keepdims=True))  # step 4
    dy = dz                                                          # step 3
    dx = dy * scale                                                  # step 2
    dq = dx @ kh                                                     # step 1, w.r.t. q
    dk = dx.T @ qh                                                   # step 1, w.r.t. k
    return dq, dk, dv


def attention_bwd(q, k, v, dout, scale: float, causal: bool):
    """Gradients (dq, dk, dv), each float64 [B, H, S, D], of the forward for
    q, k, v, dout of shape [B, H, S, D].  Holds one [S, S] matrix per head at a
    time: meant for S up to a few thousand."""
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    if q.ndim != 4 or any(x.shape != q.shape for x in (k, v, dout)):
        raise ValueError("q, k, v, dout must all have shape [B, H, S, D]")
    B, H = q.shape[:2]
    dq, dk, dv = (np.empty_like(q) for _ in range(3))
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = _head_bwd(q[b, h], k[b, h], v[b, h], dout[b, h],
                                                     float(scale), causal)
    return dq, dk, dv


def attention_bwd_rows(q, k, v, dout, scale: float, causal: bool, b: int, h: int,
                       q_rows, kv_rows):
    """Selected gradient rows of one (batch, head) at any S.

    Returns ``(dq[q_rows], dk[kv_rows], dv[kv_rows])`` as float64 arrays.  The
    forward runs over every query row to get out_i and the logsumexp lse_i;
    then attn_ij = exp(scale·q_i·k_j − lse_i) (the softmax of step 4 written
    with its normaliser), masked entries 0, and rowsum(attn ⊙ dattn)_i =
    dout_i · out_i.  A dq row then takes one row of attn, a dk or dv row one
    column.
    """
    qh, kh, vh, dh = (np.asarray(x[b, h], dtype=np.float64) for x in (q, k, v, dout))
    S = qh.shape[0]
    scale = float(scale)
    out = np.empty_like(qh)
    lse = np.empty(S)
    for r0 in range(0, S, _ROW_CHUNK):
        rows = np.arange(r0, min(S, r0 + _ROW_CHUNK))
        out[rows], lse[rows] = _head_rows(qh, kh, vh, rows, scale, causal)
    delta = np.sum(dh * out, axis=1)              # rowsum(attn ⊙ dattn), per query row
    live = np.isfinite(lse)

    q_rows = np.asarray(q_rows, dtype=np.int64)
    kv_rows = np.asarray(kv_rows, dtype=np.int64)
    # dq rows: a row of attn over all keys
    s = _scores(qh[q_rows], kh, scale, causal, q_rows)
    with np.errstate(invalid="ignore"):
        attn = np.where(live[q_rows, None], np.exp(s - lse[q_rows, None]), 0.0)
    dattn = dh[q_rows] @ vh.T
    dz = attn * (dattn - delta[q_rows, None])
    dq = (dz * scale) @ kh
    # dk, dv rows: a column of attn over all queries
    sc = (qh @ kh[kv_rows].T) * scale
    if causal:
        sc = np.where(causal_mask(S, S, cols=kv_rows), -np.inf, sc)
    with np.errstate(invalid="ignore"):
        attn_c = np.where(live[:, None], np.exp(sc - lse[:, None]), 0.0)   # [S, n]
    dv = attn_c.T @ dh
    dattn_c = dh @ vh[kv_rows].T                                           # [S, n]
    dz_c = attn_c * (dattn_c - delta[:, None])
    dk = (dz_c * scale).T @ qh
    return dq, dk, dv
