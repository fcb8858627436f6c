"""Pins for the fp64 oracle: checked against things other than itself.

Every test here runs on the CPU.  The pins are chosen so that a plausible slip
in the oracle (a dropped scale, the mask pointing the wrong way, a transposed
operand, a missing max shift, a natural/base-2 mix-up in the logsumexp) fails
at least one of them:

* hand-worked golden examples (``tests/golden``),
* a pure-Python brute force on tiny inputs,
* closed forms and invariants of the definition,
* a library routine the definition reduces to (torch's fp64 CPU SDPA).
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import (attention_fwd, attention_fwd_loops, attention_rows,
                    attention_weights, causal_mask, softmax_rows)

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


@pytest.mark.parametrize("name", ["hand_worked_s3_d2.txt", "hand_worked_peaked_s2_d1.txt"])
@pytest.mark.parametrize("causal", [True, False])
def test_golden_hand_worked(name, causal):
    g = _load_golden(name)
    out, lse = attention_fwd(_bhsd(g["q"]), _bhsd(g["k"]), _bhsd(g["v"]), g["scale"], causal)
    tag = "causal" if causal else "noncausal"
    np.testing.assert_allclose(out[0, 0], np.asarray(g[tag + "_out"], float), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], np.asarray(g[tag + "_lse"], float), rtol=1e-15, atol=1e-12)
    # the brute force agrees with the same hand-worked values
    bo, bl = attention_fwd_loops(_bhsd(g["q"]).tolist(), _bhsd(g["k"]).tolist(),
                                 _bhsd(g["v"]).tolist(), g["scale"], causal)
    np.testing.assert_allclose(np.asarray(bo)[0, 0], np.asarray(g[tag + "_out"], float), atol=1e-12)
    np.testing.assert_allclose(np.asarray(bl)[0, 0], np.asarray(g[tag + "_lse"], float), atol=1e-12)


def _rand(rng, shape, std=1.0):
    return rng.standard_normal(shape) * std


@pytest.mark.parametrize("seed", range(12))
def test_numpy_oracle_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 3))
    S, D = int(rng.integers(1, 9)), int(rng.integers(1, 5))
    causal = bool(seed % 2)
    std = [1.0, 3.0, 10.0][seed % 3]  # includes large-logit rows
    q, k, v = (_rand(rng, (B, H, S, D), std), _rand(rng, (B, H, S, D), std),
               _rand(rng, (B, H, S, D)))
    scale = float(np.float32(1 / math.sqrt(D)))
    out, lse = attention_fwd(q, k, v, scale, causal)
    bo, bl = attention_fwd_loops(q.tolist(), k.tolist(), v.tolist(), scale, causal)
    np.testing.assert_allclose(out, np.asarray(bo), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.asarray(bl), rtol=1e-14, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_weight_rows_sum_to_one_and_causal_zeros(causal):
    rng = np.random.default_rng(7)
    q, k = _rand(rng, (2, 3, 17, 8), 2.0), _rand(rng, (2, 3, 17, 8), 2.0)
    w = attention_weights(q, k, 0.35, causal)
    np.testing.assert_allclose(w.sum(-1), 1.0, atol=1e-13)
    assert (w >= 0).all()
    if causal:
        upper = np.triu(np.ones((17, 17), bool), 1)
        assert (w[..., upper] == 0).all()
        assert (w[..., ~upper] > 0).all()
    else:
        assert (w > 0).all()


def test_causal_first_row_is_v0():
    rng = np.random.default_rng(3)
    q, k, v = (_rand(rng, (2, 2, 9, 5)) for _ in range(3))
    scale = 0.41
    out, lse = attention_fwd(q, k, v, scale, True)
    assert np.array_equal(out[:, :, 0], v[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], scale * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]),
                               rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
def test_constant_v_rows_give_constant_out(causal):
    rng = np.random.default_rng(4)
    q, k = _rand(rng, (1, 2, 13, 6), 3.0), _rand(rng, (1, 2, 13, 6), 3.0)
    c = np.array([0.5, -2.0, 3.25, 0.0, 1.0, -7.5])
    v = np.broadcast_to(c, (1, 2, 13, 6)).copy()
    out, _ = attention_fwd(q, k, v, 0.4, causal)
    np.testing.assert_allclose(out, np.broadcast_to(c, out.shape), rtol=0, atol=1e-12)


@pytest.mark.parametrize("zero", ["q", "scale"])
def test_uniform_weights_when_scores_vanish(zero):
    rng = np.random.default_rng(5)
    S = 11
    q, k, v = (_rand(rng, (1, 1, S, 4)) for _ in range(3))
    scale = 0.7
    if zero == "q":
        q = np.zeros_like(q)
    else:
        scale = 0.0
    out, lse = attention_fwd(q, k, v, scale, True)
    for i in range(S):
        np.testing.assert_allclose(out[0, 0, i], v[0, 0, :i + 1].mean(0), atol=1e-13)
        np.testing.assert_allclose(lse[0, 0, i], math.log(i + 1), atol=1e-13)
    out, lse = attention_fwd(q, k, v, scale, False)
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(v[0, 0].mean(0), (S, 4)), atol=1e-13)
    np.testing.assert_allclose(lse, math.log(S), atol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
def test_single_key(causal):
    rng = np.random.default_rng(6)
    q, k, v = (_rand(rng, (3, 2, 1, 7)) for _ in range(3))
    out, lse = attention_fwd(q, k, v, 0.3, causal)
    assert np.array_equal(out, v)
    np.testing.assert_allclose(lse[..., 0], 0.3 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]),
                               atol=1e-13)


def test_noncausal_kv_permutation_equivariance():
    rng = np.random.default_rng(8)
    q, k, v = (_rand(rng, (2, 2, 19, 8), 2.0) for _ in range(3))
    perm = rng.permutation(19)
    o1, l1 = attention_fwd(q, k, v, 0.3, False)
    o2, l2 = attention_fwd(q, k[:, :, perm], v[:, :, perm], 0.3, False)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


def test_noncausal_q_permutation_permutes_out():
    rng = np.random.default_rng(9)
    q, k, v = (_rand(rng, (1, 3, 16, 4)) for _ in range(3))
    perm = rng.permutation(16)
    o1, l1 = attention_fwd(q, k, v, 0.5, False)
    o2, l2 = attention_fwd(q[:, :, perm], k, v, 0.5, False)
    np.testing.assert_allclose(o1[:, :, perm], o2, atol=1e-13)
    np.testing.assert_allclose(l1[:, :, perm], l2, atol=1e-13)


def test_causal_rows_ignore_later_keys():
    rng = np.random.default_rng(10)
    S = 20
    q, k, v = (_rand(rng, (1, 2, S, 8)) for _ in range(3))
    o1, l1 = attention_fwd(q, k, v, 0.35, True)
    for i in (0, 5, 13):
        k2, v2 = k.copy(), v.copy()
        k2[:, :, i + 1:] = _rand(rng, k2[:, :, i + 1:].shape, 5.0)
        v2[:, :, i + 1:] = _rand(rng, v2[:, :, i + 1:].shape, 5.0)
        o2, l2 = attention_fwd(q, k2, v2, 0.35, True)
        np.testing.assert_allclose(o1[:, :, :i + 1], o2[:, :, :i + 1], atol=1e-14)
        np.testing.assert_allclose(l1[:, :, :i + 1], l2[:, :, :i + 1], atol=1e-14)
        # and a later row does depend on them
        assert not np.allclose(o1[:, :, i + 1:], o2[:, :, i + 1:])


@pytest.mark.parametrize("causal", [True, False])
def test_v_shift_and_k_shift(causal):
    rng = np.random.default_rng(11)
    q, k, v = (_rand(rng, (2, 1, 14, 6)) for _ in range(3))
    scale = 0.45
    o, l = attention_fwd(q, k, v, scale, causal)
    o2, l2 = attention_fwd(q, k, v + 1.75, scale, causal)
    np.testing.assert_allclose(o2, o + 1.75, atol=1e-12)
    np.testing.assert_allclose(l2, l, atol=0)
    u = rng.standard_normal(6)
    o3, l3 = attention_fwd(q, k + u, v, scale, causal)
    np.testing.assert_allclose(o3, o, atol=1e-12)
    np.testing.assert_allclose(l3, l + scale * (q @ u), atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_matches_torch_fp64_cpu_sdpa(causal):
    """Library special case: torch's CPU fp64 SDPA computes the same definition."""
    rng = np.random.default_rng(12)
    q, k, v = (_rand(rng, (2, 3, 37, 16), 2.0) for _ in range(3))
    scale = float(np.float32(0.25))
    out, _ = attention_fwd(q, k, v, scale, causal)
    t = [torch.from_numpy(x) for x in (q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(*t, is_causal=causal, scale=scale)
    np.testing.assert_allclose(out, ref.numpy(), atol=1e-12)
    s = torch.from_numpy(q) @ torch.from_numpy(k).transpose(-1, -2) * scale
    if causal:
        s = s.masked_fill(torch.ones(37, 37, dtype=torch.bool).triu(1), float("-inf"))
    _, lse = attention_fwd(q, k, v, scale, causal)
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), atol=1e-12)


def test_large_logits_stay_finite():
    rng = np.random.default_rng(13)
    q, k, v = _rand(rng, (1, 1, 32, 8), 40.0), _rand(rng, (1, 1, 32, 8), 40.0), _rand(rng, (1, 1, 32, 8))
    out, lse = attention_fwd(q, k, v, 1.0, False)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert lse.max() > 700  # exp of these scores would overflow without the max shift


def test_safe_softmax_rule_for_fully_masked_row():
    s = np.array([[0.0, 1.0], [-np.inf, -np.inf]])
    w, lse = softmax_rows(s)
    np.testing.assert_allclose(w[0], np.exp([0.0, 1.0]) / np.exp([0.0, 1.0]).sum())
    assert (w[1] == 0).all() and lse[1] == -np.inf
    bo, bl = attention_fwd_loops([[[[0.0]]]], [[[[0.0]]]], [[[[1.0]]]], 1.0, False)
    assert bo[0][0][0] == [1.0]


def test_rows_form_equals_full_form():
    rng = np.random.default_rng(14)
    q, k, v = (_rand(rng, (2, 3, 40, 8)) for _ in range(3))
    for causal in (True, False):
        out, lse = attention_fwd(q, k, v, 0.3, causal)
        idx = np.stack([rng.integers(0, 2, 50), rng.integers(0, 3, 50), rng.integers(0, 40, 50)], 1)
        ro, rl = attention_rows(q, k, v, 0.3, causal, idx)
        np.testing.assert_array_equal(ro, out[idx[:, 0], idx[:, 1], idx[:, 2]])
        np.testing.assert_array_equal(rl, lse[idx[:, 0], idx[:, 1], idx[:, 2]])


# ------------------------------------------------------------------ planted mistakes
# Forward variants with one plausible slip each; every one must fail at least
# one of the pins above (the golden examples, the brute force, torch's SDPA,
# the first causal row, finiteness at large logits).


def _fwd_mutant(kind):
    def fwd(q, k, v, scale, causal):
        q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
        B, H, S, D = q.shape
        out = np.empty_like(q)
        lse = np.empty((B, H, S))
        for b in range(B):
            for h in range(H):
                kh = k[b, h][::-1] if kind == "k_reversed" else k[b, h]
                vh = v[b, h][::-1] if kind == "v_reversed" else v[b, h]
                s = q[b, h] @ kh.T
                if kind != "scale_dropped":
                    s = s * scale
                if causal:
                    i, j = np.arange(S)[:, None], np.arange(S)[None, :]
                    s = np.where((j < i) if kind == "mask_reversed" else (j > i), -np.inf, s)
                m = 0.0 if kind == "no_max_shift" else np.max(s, axis=1, keepdims=True)
                with np.errstate(over="ignore", invalid="ignore"):
                    p = np.exp(s - m)
                    l = p.sum(axis=1, keepdims=True)
                    out[b, h] = (p / l) @ vh
                    lse[b, h] = ((m + (np.log2(l) if kind == "lse_log2" else np.log(l)))[:, 0])
        return out, lse
    return fwd


def _fwd_pins(fwd):
    """The forward pins as checks over an implementation; False if any fails."""
    for name in ("hand_worked_s3_d2.txt", "hand_worked_peaked_s2_d1.txt"):
        g = _load_golden(name)
        for causal, tag in ((True, "causal"), (False, "noncausal")):
            out, lse = fwd(_bhsd(g["q"]), _bhsd(g["k"]), _bhsd(g["v"]), g["scale"], causal)
            if not (np.allclose(out[0, 0], np.asarray(g[tag + "_out"], float), atol=1e-12)
                    and np.allclose(lse[0, 0], np.asarray(g[tag + "_lse"], float), atol=1e-12)):
                return False
    rng = np.random.default_rng(31)
    q, k, v = (_rand(rng, (1, 2, 6, 3), 2.0) for _ in range(3))
    for causal in (True, False):
        out, lse = fwd(q, k, v, 0.6, causal)
        bo, bl = attention_fwd_loops(q.tolist(), k.tolist(), v.tolist(), 0.6, causal)
        if not (np.allclose(out, np.asarray(bo), atol=1e-12) and np.allclose(lse, np.asarray(bl), atol=1e-12)):
            return False
    return True


_FWD_MUTANTS = ["mask_reversed", "scale_dropped", "k_reversed", "v_reversed", "lse_log2",
                "no_max_shift"]


def test_forward_mutant_harness_unmutated_passes():
    assert _fwd_pins(_fwd_mutant("none"))
    assert _fwd_pins(attention_fwd)


@pytest.mark.parametrize("kind", _FWD_MUTANTS)
def test_forward_planted_mistake_fails_a_pin(kind):
    assert not _fwd_pins(_fwd_mutant(kind)), kind


# ------------------------------------------------------------------ the causal mask
# "Math backend" section of the profiling post: the mask is built as a matrix
# of ones whose lower triangle is kept (tril), and the positions outside it
# are filled with −inf.  The pins below rebuild that construction with
# numpy's tril (a library routine, not the oracle's index comparison), spell
# out one small case by hand, and check the row/column blocks the row forms
# of the oracle use against the full mask.


def _mask_pins(fn):
    """The causal-mask pins as checks over an implementation; False if any fails."""
    hand = np.array([[False, True, True],
                     [False, False, True],
                     [False, False, False]])
    if not np.array_equal(fn(3, 3), hand):
        return False
    for s_q, s_k in ((1, 1), (1, 5), (5, 1), (4, 7), (7, 4), (16, 16)):
        tril_kept = np.tril(np.ones((s_q, s_k), dtype=bool))
        m = fn(s_q, s_k)
        if m.shape != (s_q, s_k) or not np.array_equal(m, ~tril_kept):
            return False
    rows, cols = np.array([6, 0, 3]), np.array([5, 1, 6, 2])
    full = fn(7, 7)
    if not (np.array_equal(fn(7, 7, rows=rows), full[rows])
            and np.array_equal(fn(7, 7, cols=cols), full[:, cols])
            and np.array_equal(fn(7, 7, rows=rows, cols=cols), full[np.ix_(rows, cols)])):
        return False
    return True


def test_causal_mask_is_the_complement_of_tril():
    assert _mask_pins(causal_mask)


def test_causal_mask_rejects_rows_outside_the_matrix():
    with pytest.raises(ValueError):
        causal_mask(4, 4, rows=[4])
    with pytest.raises(ValueError):
        causal_mask(4, 4, cols=[-1])


def _mask_mutant(kind):
    def fn(s_q, s_k, rows=None, cols=None):
        i = np.arange(s_q) if rows is None else np.asarray(rows)
        j = np.arange(s_k) if cols is None else np.asarray(cols)
        if kind == "diagonal_masked":
            return j[None, :] >= i[:, None]
        if kind == "direction_reversed":
            return j[None, :] < i[:, None]
        if kind == "bottom_right_aligned":
            return j[None, :] > i[:, None] + (s_k - s_q)
        if kind == "rows_ignored":
            return j[None, :] > np.arange(i.size)[:, None]
        return j[None, :] > i[:, None]
    return fn


def test_mask_mutant_harness_unmutated_passes():
    assert _mask_pins(_mask_mutant("none"))


@pytest.mark.parametrize("kind", ["diagonal_masked", "direction_reversed", "bottom_right_aligned",
                                  "rows_ignored"])
def test_mask_planted_mistake_fails_a_pin(kind):
    assert not _mask_pins(_mask_mutant(kind)), kind


def test_forward_uses_the_pinned_mask(monkeypatch):
    """The forward's step 3 goes through causal_mask: a slip planted there
    shows up in the forward's own pins (brute force, hand-worked values)."""
    import oracle.attention as oa
    assert _fwd_pins(attention_fwd)
    monkeypatch.setattr(oa, "causal_mask", _mask_mutant("diagonal_masked"))
    q = np.arange(6, dtype=np.float64).reshape(1, 1, 3, 2) / 5
    with np.errstate(invalid="ignore"):
        out, _ = oa.attention_fwd(q, q, q, 1.0, True)
    bo, _ = attention_fwd_loops(q.tolist(), q.tolist(), q.tolist(), 1.0, True)
    assert not np.allclose(out, np.asarray(bo), equal_nan=False)
