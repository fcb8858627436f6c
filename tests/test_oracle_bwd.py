"""Pins for the fp64 backward oracle, checked against things other than itself.

Each pin is a check over an implementation ``bwd(q, k, v, dout, scale,
causal) -> (dq, dk, dv)``, so that the same checks run on the oracle and on
planted mistakes (a dropped scale, a missing transpose, a wrong sign, the
rowsum term left out, the mask reversed): every planted mistake must fail at
least one pin.

* a hand-worked example (``tests/golden/bwd_hand_worked_s2_d1.txt``),
* central finite differences of L = Σ dout ⊙ out through the pinned forward
  oracle,
* torch fp64 autograd through a separately written five-step forward,
* invariants: Σ_j dk_j = 0 (each row of dz sums to 0), Σ_j dv_j = Σ_i dout_i
  (each row of attn sums to 1), dq unchanged by a constant shift of every key,
* a single key: dv = dout, dq = dk = 0.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention_bwd, attention_bwd_rows, attention_fwd
from oracle.attention import _scores, softmax_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_golden(name):
    ns = {"__builtins__": {}, "ln": math.log}
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, expr = line.split("=", 1)
            vals[key.strip()] = eval(expr, ns)  # fixture values are plain expressions
    return vals


def _bhsd(x):
    return np.asarray(x, dtype=np.float64)[None, None]


def _rand(rng, shape, std=1.0):
    return rng.standard_normal(shape) * std


# ------------------------------------------------------------------ pins


def pin_golden(bwd):
    g = _load_golden("bwd_hand_worked_s2_d1.txt")
    for causal, tag in ((True, "causal"), (False, "noncausal")):
        dq, dk, dv = bwd(_bhsd(g["q"]), _bhsd(g["k"]), _bhsd(g["v"]), _bhsd(g["dout"]),
                         g["scale"], causal)
        for got, key in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
            if not np.allclose(got[0, 0], np.asarray(g[f"{tag}_{key}"]), rtol=0, atol=1e-12):
                return False
    return True


def pin_finite_differences(bwd):
    rng = np.random.default_rng(21)
    shape = (1, 2, 5, 3)
    q, k, v, dout = (_rand(rng, shape) for _ in range(4))
    scale, eps = 0.7, 1e-5
    for causal in (True, False):
        dq, dk, dv = bwd(q, k, v, dout, scale, causal)

        def loss(qq, kk, vv):
            return float(np.sum(dout * attention_fwd(qq, kk, vv, scale, causal)[0]))

        for which, grad in ((0, dq), (1, dk), (2, dv)):
            args = [q, k, v]
            num = np.empty(shape)
            for idx in np.ndindex(*shape):
                plus = [a.copy() for a in args]
                minus = [a.copy() for a in args]
                plus[which][idx] += eps
                minus[which][idx] -= eps
                num[idx] = (loss(*plus) - loss(*minus)) / (2 * eps)
            if not np.allclose(grad, num, rtol=1e-6, atol=1e-8):
                return False
    return True


def _torch_forward(q, k, v, scale, causal):
    """The five steps written again in torch, for autograd (independent of the oracle)."""
    s = torch.matmul(q, k.transpose(-2, -1)) * scale
    if causal:
        n = s.shape[-1]
        keep = torch.ones(n, n, dtype=torch.bool).tril()
        s = s.masked_fill(~keep, float("-inf"))
    return torch.matmul(torch.softmax(s, dim=-1), v)


def pin_torch_autograd(bwd):
    rng = np.random.default_rng(22)
    shape = (2, 3, 17, 8)
    q, k, v, dout = (_rand(rng, shape, 1.5) for _ in range(4))
    for causal in (True, False):
        tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
        _torch_forward(tq, tk, tv, 0.4, causal).backward(torch.tensor(dout, dtype=torch.float64))
        dq, dk, dv = bwd(q, k, v, dout, 0.4, causal)
        for got, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
            if not np.allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12):
                return False
    return True


def pin_invariants(bwd):
    rng = np.random.default_rng(23)
    shape = (1, 2, 12, 4)
    q, k, v, dout = (_rand(rng, shape) for _ in range(4))
    shift = _rand(rng, (1, 1, 1, 4))
    for causal in (True, False):
        dq, dk, dv = bwd(q, k, v, dout, 0.8, causal)
        if not np.allclose(dk.sum(axis=2), 0.0, atol=1e-12):
            return False
        if not np.allclose(dv.sum(axis=2), dout.sum(axis=2), rtol=1e-12, atol=1e-12):
            return False
        dq2, _, _ = bwd(q, k + shift, v, dout, 0.8, causal)
        if not np.allclose(dq2, dq, rtol=1e-10, atol=1e-12):
            return False
    return True


def pin_single_key(bwd):
    rng = np.random.default_rng(24)
    q, k, v, dout = (_rand(rng, (2, 2, 1, 5)) for _ in range(4))
    for causal in (True, False):
        dq, dk, dv = bwd(q, k, v, dout, 0.9, causal)
        if not (np.allclose(dv, dout, atol=1e-14) and np.allclose(dq, 0, atol=1e-14)
                and np.allclose(dk, 0, atol=1e-14)):
            return False
    return True


PINS = [pin_golden, pin_finite_differences, pin_torch_autograd, pin_invariants, pin_single_key]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_passes_pin(pin):
    assert pin(attention_bwd)


# ------------------------------------------------------------------ planted mistakes


def _mutant(kind):
    """The oracle's five reversed steps with one plausible slip planted."""

    def bwd(q, k, v, dout, scale, causal):
        q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
        out = [np.empty_like(q) for _ in range(3)]
        for b in range(q.shape[0]):
            for h in range(q.shape[1]):
                qh, kh, vh, dh = q[b, h], k[b, h], v[b, h], dout[b, h]
                S = qh.shape[0]
                rows = np.arange(S)
                s = _scores(qh, kh, scale, False, rows)
                if causal:
                    j = np.arange(S)[None, :]
                    bad = j < rows[:, None] if kind == "mask_reversed" else j > rows[:, None]
                    s = np.where(bad, -np.inf, s)
                attn, _ = softmax_rows(s)
                dattn = dh @ vh.T
                dv = (attn @ dh) if kind == "dv_no_transpose" else (attn.T @ dh)
                rs = np.sum(attn * dattn, axis=1, keepdims=True)
                if kind == "rowsum_dropped":
                    dz = attn * dattn
                elif kind == "rowsum_sign":
                    dz = attn * (dattn + rs)
                else:
                    dz = attn * (dattn - rs)
                dx = dz if kind == "scale_dropped" else dz * scale
                dq = dx @ kh
                dk = (dx @ qh) if kind == "dk_no_transpose" else (dx.T @ qh)
                if kind == "dq_uses_v":
                    dq = dx @ vh
                out[0][b, h], out[1][b, h], out[2][b, h] = dq, dk, dv
        return tuple(out)

    return bwd


MUTANTS = ["mask_reversed", "dv_no_transpose", "rowsum_dropped", "rowsum_sign", "scale_dropped",
           "dk_no_transpose", "dq_uses_v"]


def test_unmutated_copy_passes_every_pin():
    """The mutant harness without a slip is the oracle: every pin holds."""
    bwd = _mutant("none")
    assert all(pin(bwd) for pin in PINS)


@pytest.mark.parametrize("kind", MUTANTS)
def test_planted_mistake_fails_a_pin(kind):
    bwd = _mutant(kind)
    assert not all(pin(bwd) for pin in PINS), kind


# ------------------------------------------------------------------ row form


def test_rows_form_equals_full_form():
    rng = np.random.default_rng(25)
    q, k, v, dout = (_rand(rng, (2, 2, 70, 8)) for _ in range(4))
    for causal in (True, False):
        dq, dk, dv = attention_bwd(q, k, v, dout, 0.35, causal)
        qr = np.array([0, 1, 33, 69])
        kr = np.array([0, 5, 64, 69])
        rq, rk, rv = attention_bwd_rows(q, k, v, dout, 0.35, causal, 1, 1, qr, kr)
        np.testing.assert_allclose(rq, dq[1, 1, qr], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(rk, dk[1, 1, kr], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(rv, dv[1, 1, kr], rtol=1e-12, atol=1e-13)


def test_large_logits_stay_finite():
    rng = np.random.default_rng(26)
    q, k, v, dout = (_rand(rng, (1, 1, 9, 4), 30.0) for _ in range(4))
    for causal in (True, False):
        for g in attention_bwd(q, k, v, dout, 1.0, causal):
            assert np.isfinite(g).all()
