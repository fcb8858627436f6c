"""fp64 CPU oracle for the fused attention forward and its gradient.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product library never does, and the two share no code.
"""
from .attention import (attention_fwd, attention_rows, attention_weights,
                        causal_mask, softmax_rows)
from .attention_bwd import attention_bwd, attention_bwd_rows
from .brute import attention_fwd_loops

__all__ = ["attention_fwd", "attention_rows", "attention_weights", "causal_mask",
           "softmax_rows", "attention_fwd_loops", "attention_bwd", "attention_bwd_rows"]
