"""Seeded synthetic workloads shared by the tests, the smoke check and the bench.

This module only draws inputs and names shapes; it holds none of the attention
arithmetic, so both the CUDA path and the fp64 oracle can be fed from it
without sharing any computation.

Recipe (the same for every workload): a CPU ``torch.Generator`` seeded with
``seed`` (0 unless a caller says otherwise) draws q, k and v with
``torch.randn`` in that order as float32 of shape [B, H, S, D]; q and k are
multiplied by ``qk_std`` and v by ``v_std``; each is then rounded to bfloat16
(round-to-nearest-even).  The oracle reads these same bf16 values, converted
exactly to float64.  scale defaults to float32(1/√D), the value the
``NaiveCausalAttention`` module of "Profiling in PyTorch (Part 3): Attention is
all you profile" uses.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

__all__ = ["Workload", "WORKLOADS", "default_scale", "make_qkv", "check_rows",
           "counted_flops", "algorithmic_bytes"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    D: int
    causal: bool
    qk_std: float = 1.0
    v_std: float = 1.0
    about: str = ""

    @property
    def shape(self):
        return (self.B, self.H, self.S, self.D)


WORKLOADS = {
    "c1": Workload("c1", 1, 2, 128, 64, True,
                   about="causal B=1 H=2 S=128 D=64, N(0,1)"),
    "c2": Workload("c2", 4, 16, 1024, 64, True,
                   about="causal B=4 H=16 S=1024 D=64, N(0,1)"),
    "c3": Workload("c3", 2, 16, 4096, 128, True,
                   about="causal B=2 H=16 S=4096 D=128, N(0,1)"),
    "c4": Workload("c4", 8, 16, 2048, 128, False, qk_std=3.0,
                   about="non-causal B=8 H=16 S=2048 D=128, q,k N(0,3^2), v N(0,1)"),
    "c5": Workload("c5", 1, 32, 16384, 128, True,
                   about="causal long-context B=1 H=32 S=16384 D=128, N(0,1)"),
}


def default_scale(D: int) -> float:
    """float32(1/sqrt(D)) as a Python float (exactly representable in fp32)."""
    return float(np.float32(1.0 / math.sqrt(D)))


def make_qkv(w: Workload | tuple, seed: int = 0, qk_std: float | None = None,
             v_std: float | None = None, dtype: torch.dtype = torch.bfloat16):
    """Draw (q, k, v) as contiguous CPU tensors of shape [B, H, S, D], rounded
    to ``dtype`` (bf16 by default, or fp16).

    ``w`` is a Workload or a (B, H, S, D) tuple (then N(0,1) unless stds given).
    """
    if isinstance(w, Workload):
        shape = w.shape
        qs = w.qk_std if qk_std is None else qk_std
        vs = w.v_std if v_std is None else v_std
    else:
        shape = tuple(int(x) for x in w)
        qs = 1.0 if qk_std is None else qk_std
        vs = 1.0 if v_std is None else v_std
    g = torch.Generator().manual_seed(int(seed))
    out = []
    for std in (qs, qs, vs):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        out.append(x.to(dtype).contiguous())
    return tuple(out)


def check_rows(w: Workload) -> np.ndarray:
    """(b, h, i) triples compared against the oracle for a workload, [n, 3] int64.

    c1, c2, c4: every row.  c3: every row of heads (0, 0) and (1, 15) plus 256
    rows drawn by ``numpy.random.default_rng(1)`` from the other heads.  c5: rows
    0 and S-1 of every head plus 448 rows drawn by ``default_rng(2)``.
    """
    B, H, S = w.B, w.H, w.S
    if w.name == "c3":
        full = [(0, 0), (1, 15)]
        rows = [(b, h, i) for (b, h) in full for i in range(S)]
        rng = np.random.default_rng(1)
        others = [(b, h) for b in range(B) for h in range(H) if (b, h) not in full]
        pick = rng.integers(0, len(others), size=256)
        ii = rng.integers(0, S, size=256)
        rows += [(others[p][0], others[p][1], int(i)) for p, i in zip(pick, ii)]
        return np.asarray(rows, dtype=np.int64)
    if w.name == "c5":
        rows = [(0, h, i) for h in range(H) for i in (0, S - 1)]
        rng = np.random.default_rng(2)
        hh = rng.integers(0, H, size=448)
        ii = rng.integers(0, S, size=448)
        rows += [(0, int(h), int(i)) for h, i in zip(hh, ii)]
        return np.asarray(rows, dtype=np.int64)
    b, h, i = np.meshgrid(np.arange(B), np.arange(H), np.arange(S), indexing="ij")
    return np.stack([b.ravel(), h.ravel(), i.ravel()], axis=1).astype(np.int64)


def counted_flops(B: int, H: int, S: int, D: int, causal: bool) -> int:
    """Counted FLOPs of one forward: 4·B·H·S²·D, halved under a causal mask."""
    full = 4 * B * H * S * S * D
    return full // 2 if causal else full


def algorithmic_bytes(B: int, H: int, S: int, D: int) -> int:
    """HBM bytes a forward must move at least: q, k, v read + out written (bf16), lse (fp32)."""
    return 4 * B * H * S * D * 2 + 4 * B * H * S
