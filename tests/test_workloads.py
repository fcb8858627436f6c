"""Host-side checks of the seeded input generators and of code independence."""
import os
import re

import numpy as np
import torch

from exact_attention_68_gb300.workloads import (WORKLOADS, check_rows, counted_flops,
                                                default_scale, make_qkv)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_generator_is_seeded_and_bf16():
    q1, k1, v1 = make_qkv((1, 2, 33, 64), seed=0)
    q2, k2, v2 = make_qkv((1, 2, 33, 64), seed=0)
    q3, _, _ = make_qkv((1, 2, 33, 64), seed=1)
    for a, b in ((q1, q2), (k1, k2), (v1, v2)):
        assert a.dtype == torch.bfloat16 and a.is_contiguous() and a.shape == (1, 2, 33, 64)
        assert torch.equal(a, b)
    assert not torch.equal(q1, q3)
    assert not torch.equal(q1, k1)


def test_qk_std_scales_only_q_and_k():
    q, k, v = make_qkv(WORKLOADS["c4"].__class__("t", 1, 1, 4096, 128, False, qk_std=3.0))
    assert 2.8 < q.float().std().item() < 3.2 and 2.8 < k.float().std().item() < 3.2
    assert 0.9 < v.float().std().item() < 1.1


def test_check_rows_counts():
    assert check_rows(WORKLOADS["c1"]).shape == (256, 3)
    assert check_rows(WORKLOADS["c3"]).shape == (2 * 4096 + 256, 3)
    r5 = check_rows(WORKLOADS["c5"])
    assert r5.shape == (512, 3)
    assert {0, 16383} <= set(r5[:, 2].tolist())
    for w in WORKLOADS.values():
        r = check_rows(w)
        assert (r[:, 0] < w.B).all() and (r[:, 1] < w.H).all() and (r[:, 2] < w.S).all()


def test_counted_flops_and_scale():
    assert counted_flops(1, 32, 16384, 128, True) == 2 * 32 * 16384 ** 2 * 128
    assert counted_flops(8, 16, 2048, 128, False) == 4 * 8 * 16 * 2048 ** 2 * 128
    assert default_scale(64) == 0.125
    assert default_scale(128) == float(np.float32(1 / np.sqrt(128)))


def _py_imports(path):
    with open(path) as f:
        src = f.read()
    return set(re.findall(r"^\s*(?:from|import)\s+([\w\.]+)", src, re.M))


def test_oracle_and_product_share_no_code():
    for dirpath, _, files in os.walk(os.path.join(ROOT, "oracle")):
        for f in files:
            if f.endswith(".py"):
                mods = _py_imports(os.path.join(dirpath, f))
                assert not any(m.startswith("exact_attention_68_gb300") for m in mods), f
    pkg = os.path.join(ROOT, "exact_attention_68_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            p = os.path.join(dirpath, f)
            if f.endswith(".py"):
                mods = _py_imports(p)
                assert not any(m == "oracle" or m.startswith("oracle.") for m in mods), p
            if f.endswith((".cu", ".cuh", ".h", ".cpp")):
                with open(p) as fh:
                    assert not re.search(r'#include\s*[<"][^>"]*oracle', fh.read()), p
