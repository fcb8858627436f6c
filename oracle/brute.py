"""Pure-Python brute-force attention for tiny inputs (pins the numpy oracle).

TEST INFRASTRUCTURE, like everything under ``oracle/``.

It restates the five steps of the "Naive attention" section of "Profiling in
PyTorch (Part 3): Attention is all you profile" with explicit loops,
``math.exp`` and exactly rounded sums (``math.fsum``), and shares nothing with
``oracle.attention`` beyond the definition itself: no numpy, no max-shift
helper, no mask helper.  Inputs are nested Python lists (or anything indexable)
of shape [B][H][S][D].
"""
from __future__ import annotations

import math

__all__ = ["attention_fwd_loops"]


def attention_fwd_loops(q, k, v, scale, causal):
    """Return (out, lse) as nested lists [B][H][S][D] and [B][H][S]."""
    out, lse = [], []
    for b in range(len(q)):
        ob, lb = [], []
        for h in range(len(q[b])):
            qh, kh, vh = q[b][h], k[b][h], v[b][h]
            S = len(qh)
            D = len(qh[0]) if S else 0
            oh, lh = [], []
            for i in range(S):
                scores = []
                for j in range(S):
                    if causal and j > i:
                        scores.append(-math.inf)
                    else:
                        dot = math.fsum(float(qh[i][d]) * float(kh[j][d]) for d in range(D))
                        scores.append(dot * float(scale))
                top = max(scores)
                if top == -math.inf:
                    oh.append([0.0] * D)
                    lh.append(-math.inf)
                    continue
                e = [math.exp(s - top) for s in scores]
                total = math.fsum(e)
                oh.append([math.fsum(e[j] * float(vh[j][d]) for j in range(S)) / total
                           for d in range(D)])
                lh.append(top + math.log(total))
            ob.append(oh)
            lb.append(lh)
        out.append(ob)
        lse.append(lb)
    return out, lse
