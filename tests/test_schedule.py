"""Host checks of the forward kernel's grid schedule (CTA index -> work unit).

The map is compiled from the kernel's own header into a host-only shim; the
checks need no GPU.  A work unit is one (b·H + h) slice and one unit level u
(Q tile u); under the causal mask level u costs u+1 KV tile-steps.
"""
import ctypes
import itertools

import numpy as np
import pytest

from exact_attention_68_gb300 import build


@pytest.fixture(scope="module")
def shim():
    lib = ctypes.CDLL(build.build_sched_check())
    lib.sched_map.argtypes = [ctypes.c_int] * 4 + [ctypes.POINTER(ctypes.c_int)] * 2
    lib.sched_map.restype = None
    lib.sched_plan.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                                      ctypes.POINTER(ctypes.c_int)]
    lib.sched_plan.restype = None
    return lib


def _map(lib, BH, nu, G, tail):
    n = BH * nu
    bh = np.full(n, -1, np.int32)
    u = np.full(n, -1, np.int32)
    ip = ctypes.POINTER(ctypes.c_int)
    lib.sched_map(BH, nu, G, tail, bh.ctypes.data_as(ip), u.ctypes.data_as(ip))
    return bh, u


def _plan(lib, BH, nu, S, D, causal, budget=48 << 20, sms=152):
    out = (ctypes.c_int * 2)()
    lib.sched_plan(BH, nu, S, D, int(causal), budget, sms, out)
    return out[0], out[1]


CASES = [(BH, nu, G, tail)
         for BH, nu in ((1, 1), (1, 5), (3, 1), (7, 9), (32, 64), (40, 16), (5, 33))
         for G in sorted({1, 2, 3, max(1, BH // 2), BH})
         for tail in sorted({0, 1, nu // 3, nu - 1, nu})]


@pytest.mark.parametrize("BH,nu,G,tail", CASES)
def test_map_is_a_bijection_in_range(shim, BH, nu, G, tail):
    bh, u = _map(shim, BH, nu, G, tail)
    assert bh.min() >= 0 and bh.max() < BH and u.min() >= 0 and u.max() < nu
    pairs = bh.astype(np.int64) * nu + u
    assert np.array_equal(np.sort(pairs), np.arange(BH * nu))


@pytest.mark.parametrize("BH,nu,G,tail", CASES)
def test_phase_order(shim, BH, nu, G, tail):
    """Phase 1 (levels >= tail) comes first, group by group, each group
    heaviest first with its slices side by side; phase 2 is heaviest first
    over all slices."""
    bh, u = _map(shim, BH, nu, G, tail)
    p1 = BH * (nu - tail)
    assert (u[:p1] >= tail).all() and (u[p1:] < tail).all()
    # phase 2: level-major, slices in order
    exp_u2 = np.repeat(np.arange(tail - 1, -1, -1), BH)
    exp_b2 = np.tile(np.arange(BH), tail)
    assert np.array_equal(u[p1:], exp_u2) and np.array_equal(bh[p1:], exp_b2)
    # phase 1: groups of G consecutive slices, each run to completion
    x = 0
    for g0 in range(0, BH, G):
        gs = min(G, BH - g0)
        n = gs * (nu - tail)
        exp_u = np.repeat(np.arange(nu - 1, tail - 1, -1), gs)
        exp_b = np.tile(np.arange(g0, g0 + gs), nu - tail)
        assert np.array_equal(u[x:x + n], exp_u) and np.array_equal(bh[x:x + n], exp_b)
        x += n
    assert x == p1


def test_one_group_is_plain_heaviest_first(shim):
    for tail in (0, 5, 17):
        bh, u = _map(shim, 12, 17, 12, tail)
        assert np.array_equal(u, np.repeat(np.arange(16, -1, -1), 12))
        assert np.array_equal(bh, np.tile(np.arange(12), 17))


@pytest.mark.parametrize("BH,S,D", list(itertools.product((1, 6, 32, 40, 128), (128, 1000, 4096, 16384, 131072), (64, 128))))
@pytest.mark.parametrize("causal", [True, False])
def test_plan_rules(shim, BH, S, D, causal):
    budget, sms = 48 << 20, 152
    nu = (S + 255) // 256
    G, tail = _plan(shim, BH, nu, S, D, causal, budget, sms)
    assert 1 <= G <= BH
    kv = S * D * 4
    if G > 1:
        assert G * kv <= budget  # one group's K/V stays inside the budget
    if G < BH:
        assert (G + 1) * kv > budget  # and the group is as large as the budget allows
    if not causal:
        assert tail == 0
    else:
        assert 0 <= tail <= nu
        want = nu * sms // 2
        assert tail == nu or tail * tail * BH >= want
        assert tail == 0 or (tail - 1) ** 2 * BH < want  # the smallest such tail


def test_plan_long_context_causal(shim):
    # B=1, H=32, S=16384, D=128: 8 MiB of K/V per slice -> 6 slices per group;
    # 128 Q tiles, sqrt(128 * 152 / (2 * 32)) = 17.4 -> 18 levels in phase 2
    assert _plan(shim, 32, 128, 16384, 128, True) == (6, 18)
    # B=2, H=16, S=4096, D=128: 2 MiB per slice -> 24 per group; 32 Q tiles,
    # sqrt(32 * 152 / (2 * 32)) = 8.7 -> 9 tail levels
    assert _plan(shim, 32, 32, 4096, 128, True) == (24, 9)
    # without the mask every unit costs the same: no phase 2
    assert _plan(shim, 128, 16, 2048, 128, False) == (48, 0)


@pytest.mark.parametrize("BH", [1, 2, 7, 13, 18, 32, 100])
@pytest.mark.parametrize("per_slice_mb", [1, 6, 12, 48, 200])
def test_staged_chunk_plan_covers_every_slice_once(shim, BH, per_slice_mb):
    shim.staged_plan.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                 ctypes.POINTER(ctypes.c_int64)]
    shim.staged_plan.restype = ctypes.c_int
    out = (ctypes.c_int64 * 32)()
    target, max_chunks = 48 << 20, 8
    n = shim.staged_plan(BH, per_slice_mb << 20, target, max_chunks, out)
    assert 1 <= n <= min(BH, max_chunks)
    first = [out[2 * c] for c in range(n)]
    count = [out[2 * c + 1] for c in range(n)]
    assert first[0] == 0 and all(x >= 1 for x in count)
    assert all(first[c] + count[c] == first[c + 1] for c in range(n - 1))
    assert first[-1] + count[-1] == BH
    # all but the last chunk even; the last one half an even share (>= 1)
    if n > 1:
        assert max(count[:-1]) - min(count[:-1]) <= 1
        assert count[-1] == max(1, BH // n // 2) and count[-1] <= min(count[:-1])
    else:
        assert count == [BH]
    # as many chunks as the inputs need at about `target` bytes each, capped
    want = -(-BH * (per_slice_mb << 20) // target)
    assert n == max(1, min(want, BH, max_chunks))
