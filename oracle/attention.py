"""Plain, slow, fp64 CPU oracle for exact scaled-dot-product attention (forward).

TEST INFRASTRUCTURE. Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline / reference leg of ``bench.py`` may
import or run anything under ``oracle/``. The product path (the CUDA library
and its Python binding) never calls it, and it shares no code, header, table or
helper with that path: it only receives arrays.

What it computes, step by step, follows the five primitive steps listed in
"Profiling in PyTorch (Part 3): Attention is all you profile", section "Naive
attention" (the ``NaiveCausalAttention`` module):

  1. scores = q · kᵀ
  2. scores = scores · scale
  3. scores = masked_fill(mask, −inf)           (causal mask only)
  4. attn   = softmax(scores) along the key axis
  5. out    = attn · v

Readings taken where the pages are silent or garbled (each is also listed in
the design notes of the repository):

* Mask convention: the "Math backend" section of the same page builds the
  causal mask with ``ones → tril`` and turns it into a 0/−inf bias, i.e. the
  lower triangle (key index j ≤ query index i) is kept and j > i is masked.
  (The FlashAttention-2 blog's "Causal Masking" sentence states the relation
  backwards; the tril construction is taken as authoritative.)
* Fully masked rows follow the ``_safe_softmax`` passage of the "Math backend"
  section: such a row yields weights 0 (hence output 0) instead of NaN, and its
  logsumexp is −inf.  With a causal mask and equal query/key lengths this
  cannot happen (the diagonal is always kept); the rule is still implemented.
* logsumexp (the pages never define it): the natural logarithm of
  Σ_j exp(scale · q_i · k_j) over the unmasked keys of row i.
* The softmax subtracts the row maximum before exponentiating.  This is the
  same function mathematically; it only keeps fp64 finite for large logits.
* Inputs are whatever the caller passes (bf16 values convert exactly to
  float64); nothing here rounds to bf16.

Rows are independent by definition (step 4 normalises each row on its own), so
evaluating a subset of rows, or rows in chunks, computes exactly the same
numbers as the full matrix for those rows; no reduction is reordered.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "causal_mask",
    "softmax_rows",
    "attention_weights",
    "attention_fwd",
    "attention_rows",
]

# Rows evaluated at once for one (batch, head); bounds the size of the
# [rows, S] fp64 score block held in memory.
_ROW_CHUNK = 1024


def causal_mask(s_q: int, s_k: int, rows=None, cols=None) -> np.ndarray:
    """Boolean mask, True where a score is masked (key j > query i).

    "Math backend" section: ``ones → tril`` keeps the lower triangle, so
    query i sees keys 0..i (top-left alignment when s_q != s_k).  The full
    mask is [s_q, s_k]; ``rows`` (query indices in [0, s_q)) and ``cols``
    (key indices in [0, s_k)) select a block of it without forming the rest.
    """
    i = np.arange(s_q) if rows is None else np.asarray(rows, dtype=np.int64)
    j = np.arange(s_k) if cols is None else np.asarray(cols, dtype=np.int64)
    if i.size and (i.min() < 0 or i.max() >= s_q):
        raise ValueError("query rows must lie in [0, s_q)")
    if j.size and (j.min() < 0 or j.max() >= s_k):
        raise ValueError("key columns must lie in [0, s_k)")
    return j[None, :] > i[:, None]


def softmax_rows(scores: np.ndarray):
    """Step 4 (softmax along the last axis) plus the row logsumexp, in fp64.

    Returns ``(weights, lse)``.  A row whose scores are all −inf gets weights 0
    and lse −inf ("_safe_softmax" rule, "Math backend" section).
    """
    scores = np.asarray(scores, dtype=np.float64)
    m = np.max(scores, axis=-1, keepdims=True)
    dead = ~np.isfinite(m)  # row entirely −inf
    m_safe = np.where(dead, 0.0, m)
    p = np.exp(scores - m_safe)  # exp(−inf) = 0 for masked entries
    p = np.where(dead, 0.0, p)
    l = np.sum(p, axis=-1, keepdims=True)
    l_safe = np.where(dead, 1.0, l)
    weights = p / l_safe
    with np.errstate(divide="ignore"):
        lse = np.where(dead, -np.inf, m_safe + np.log(l_safe))
    return weights, lse[..., 0]


def _scores(q_rows: np.ndarray, k: np.ndarray, scale: float, causal: bool,
            row_index: np.ndarray) -> np.ndarray:
    """Steps 1-3 for the query rows ``row_index`` of one (batch, head)."""
    s = q_rows @ k.T                      # step 1: q · kᵀ
    s = s * scale                         # step 2: · scale
    if causal:                            # step 3: masked_fill(mask, −inf)
        s = np.where(causal_mask(k.shape[0], k.shape[0], row_index), -np.inf, s)
    return s


def attention_weights(q, k, scale: float, causal: bool) -> np.ndarray:
    """The attention-weight matrix attn = softmax(masked scaled scores).

    Shape [..., S, S]; materialised in full, so meant for small S only.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    lead = q.shape[:-2]
    s_q = q.shape[-2]
    qf = q.reshape((-1,) + q.shape[-2:])
    kf = k.reshape((-1,) + k.shape[-2:])
    out = np.empty((qf.shape[0], s_q, kf.shape[1]), dtype=np.float64)
    rows = np.arange(s_q)
    for n in range(qf.shape[0]):
        w, _ = softmax_rows(_scores(qf[n], kf[n], float(scale), causal, rows))
        out[n] = w
    return out.reshape(lead + out.shape[1:])


def _head_rows(qh, kh, vh, rows, scale, causal):
    """Steps 1-5 and the logsumexp for some query rows of one (batch, head)."""
    s = _scores(qh[rows], kh, scale, causal, rows)
    w, lse = softmax_rows(s)
    out = w @ vh                          # step 5: attn · v
    return out, lse


def attention_fwd(q, k, v, scale: float, causal: bool):
    """Full forward for q, k, v of shape [B, H, S, D] (any float dtype).

    Returns ``(out, lse)``: out float64 [B, H, S, D], lse float64 [B, H, S].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if q.ndim != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all have shape [B, H, S, D]")
    B, H, S, D = q.shape
    out = np.empty((B, H, S, D), dtype=np.float64)
    lse = np.empty((B, H, S), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, S, _ROW_CHUNK):
                rows = np.arange(r0, min(S, r0 + _ROW_CHUNK))
                o, l = _head_rows(q[b, h], k[b, h], v[b, h], rows, float(scale), causal)
                out[b, h, rows] = o
                lse[b, h, rows] = l
    return out, lse


def attention_rows(q, k, v, scale: float, causal: bool, index):
    """Forward for selected rows only.

    ``index`` is an int array of shape [n, 3] holding (b, h, i) triples.
    Returns ``(out [n, D], lse [n])`` in the order of ``index``; each row is
    exactly the row the full forward would produce.
    """
    q = np.asarray(q)
    k = np.asarray(k)
    v = np.asarray(v)
    index = np.asarray(index, dtype=np.int64).reshape(-1, 3)
    D = q.shape[-1]
    out = np.empty((index.shape[0], D), dtype=np.float64)
    lse = np.empty((index.shape[0],), dtype=np.float64)
    # group the requested rows by (b, h) so each head's K and V convert once
    keys = index[:, 0] * (q.shape[1] + 1) + index[:, 1]
    for key in np.unique(keys):
        sel = np.nonzero(keys == key)[0]
        b, h = int(index[sel[0], 0]), int(index[sel[0], 1])
        kh = np.asarray(k[b, h], dtype=np.float64)
        vh = np.asarray(v[b, h], dtype=np.float64)
        qh = np.asarray(q[b, h], dtype=np.float64)
        for c0 in range(0, sel.size, _ROW_CHUNK):
            part = sel[c0:c0 + _ROW_CHUNK]
            rows = index[part, 2]
            o, l = _head_rows(qh, kh, vh, rows, float(scale), causal)
            out[part] = o
            lse[part] = l
    return out, lse
