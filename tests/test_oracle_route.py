"""Pins of the oracle's router: specified sigmoid, selection, gates, logits."""
import itertools
import math

import numpy as np
import pytest

from oracle import route as R
from oracle import sigmoid as SG


def test_exp_spec_error_bound():
    z = np.linspace(-80, 80, 400001).astype(np.float32)
    ref = np.exp(z.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    err = np.abs(SG.exp_spec(z).astype(np.float64) - ref) / ulp
    assert err.max() <= 2.0


def test_cody_waite_split():
    c1 = float(SG.C1)
    m, _ = math.frexp(c1)
    assert (m * 2 ** 9).is_integer()                       # at most 9 significant bits
    assert abs(c1 + float(SG.C2) - math.log(2.0)) < 1e-10
    for n in range(-127, 128):                              # n * C1 exact in fp32
        assert float(np.float32(n) * SG.C1) == n * c1


def test_sigmoid_special_values():
    assert SG.sigmoid_spec(np.float32(0.0)) == np.float32(0.5)
    l = np.linspace(-30, 30, 20001).astype(np.float32)
    s = SG.sigmoid_spec(l)
    assert np.all(np.diff(s.astype(np.float64)) >= 0)
    ref = 1.0 / (1.0 + np.exp(-l.astype(np.float64)))
    assert np.max(np.abs(s - ref) / np.maximum(ref, 1e-30)) < 4e-7
    assert np.max(np.abs(s.astype(np.float64) + SG.sigmoid_spec(-l) - 1.0)) < 2.5e-7
    assert SG.sigmoid_spec(np.float32(1e4)) == 1.0 and SG.sigmoid_spec(np.float32(-1e4)) > 0


def _dominates(va, a, vb, b):
    return va > vb or (va == vb and a < b)


def _brute_select(v, k, G, g_top):
    """Selection characterised by pairwise dominance, with groups by exhaustive search."""
    E = v.shape[0]
    per = E // G
    if G > 1:
        gs = []
        for g in range(G):
            vals = v[g * per:(g + 1) * per]
            gs.append(max(np.float32(vals[a] + vals[b]) for a, b in itertools.combinations(range(per), 2)))
        kept = None
        for cand in itertools.combinations(range(G), g_top):
            ok = all(_dominates(gs[a], a, gs[b], b) for a in cand for b in range(G) if b not in cand)
            if ok:
                kept = cand
        allowed = [e for e in range(E) if e // per in kept]
    else:
        allowed = list(range(E))
    chosen = None
    for cand in itertools.combinations(allowed, k):
        if all(_dominates(v[a], a, v[b], b) for a in cand for b in allowed if b not in cand):
            chosen = cand
    order = sorted(chosen, key=lambda e: (-float(v[e]), e))
    return order


def test_select_brute_force_plain_topk():
    rng = np.random.default_rng(0)
    lg = rng.normal(0, 2, (200, 8)).astype(np.float32)
    lg[:20, 3] = lg[:20, 5]                             # force score ties
    b = np.zeros(8, np.float32)
    idx, w, s = R.select(lg, b, 2, 1, 1)
    v = (SG.sigmoid_spec(lg) + b).astype(np.float32)
    for t in range(200):
        assert list(idx[t]) == _brute_select(v[t], 2, 1, 1)


def test_select_brute_force_groups():
    rng = np.random.default_rng(1)
    E, G, g_top, k = 16, 4, 2, 4
    lg = rng.normal(0, 2, (150, E)).astype(np.float32)
    b = rng.normal(0, 0.1, E).astype(np.float32)
    idx, w, s = R.select(lg, b, k, G, g_top)
    v = (SG.sigmoid_spec(lg) + b).astype(np.float32)
    for t in range(150):
        assert list(idx[t]) == _brute_select(v[t], k, G, g_top)


def test_group_stage_noop_with_one_group():
    rng = np.random.default_rng(2)
    lg = rng.normal(0, 2, (64, 32)).astype(np.float32)
    b = rng.normal(0, 0.1, 32).astype(np.float32)
    a = R.select(lg, b, 4, 1, 1)
    c = R.select(lg, b, 4, 4, 4)                        # all groups kept
    assert np.array_equal(a[0], c[0])


def test_gates_sum_to_one_and_use_unbiased_scores():
    rng = np.random.default_rng(3)
    lg = rng.normal(0, 2, (500, 64)).astype(np.float32)
    b = rng.normal(0, 0.5, 64).astype(np.float32)
    idx, w, s = R.select(lg, b, 8, 8, 4)
    tot = w.astype(np.float64).sum(axis=1)
    assert np.all(np.abs(tot - 1.0) <= 8 * 2.0 ** -24)
    assert np.all(w > 0)
    ss = SG.sigmoid_spec(lg)
    assert np.array_equal(s, np.take_along_axis(ss, idx, 1))
    ratio = w / s
    assert np.allclose(ratio, ratio[:, :1], rtol=1e-6)   # w proportional to unbiased s
    # indices distinct and inside kept groups (at most g_top groups used)
    assert all(len(set(r)) == 8 for r in idx)
    assert all(len(set((np.array(r) // 8).tolist())) <= 4 for r in idx)


def test_all_ties_pick_lowest_indices():
    lg = np.zeros((3, 16), np.float32)
    idx, w, _ = R.select(lg, np.zeros(16, np.float32), 4, 4, 2)
    assert np.array_equal(idx, np.tile(np.arange(4), (3, 1)))
    assert np.all(w == np.float32(0.25))


def test_router_logits_exact_sums():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(6, 40)).astype(np.float32)
    wr = rng.normal(0, 0.02, (5, 40)).astype(np.float32)
    lg = R.router_logits(x, wr)
    for t in range(6):
        for e in range(5):
            ref = math.fsum(float(x[t, c]) * float(wr[e, c]) for c in range(40))
            assert lg[t, e] == np.float32(ref)


def test_selection_margin_positive_for_strict_choice():
    rng = np.random.default_rng(5)
    lg = rng.normal(0, 2, (50, 16)).astype(np.float32)
    b = np.zeros(16, np.float32)
    idx, _, _ = R.select(lg, b, 2)
    assert np.all(R.selection_margin(lg, b, idx) >= 0)


def _brute_select_f64(v, k, G, g_top):
    """Dominance search as in _brute_select, with fp64 group scores."""
    E = v.shape[0]
    per = E // G
    allowed = list(range(E))
    if G > 1:
        gs = [max(v[g * per + a] + v[g * per + b] for a, b in itertools.combinations(range(per), 2))
              for g in range(G)]
        kept = next(c for c in itertools.combinations(range(G), g_top)
                    if all(_dominates(gs[a], a, gs[b], b) for a in c for b in range(G) if b not in c))
        allowed = [e for e in range(E) if e // per in kept]
    chosen = next(c for c in itertools.combinations(allowed, k)
                  if all(_dominates(v[a], a, v[b], b) for a in c for b in allowed if b not in c))
    return sorted(chosen, key=lambda e: (-float(v[e]), e))


@pytest.mark.parametrize("E,G,g_top,k", [(8, 1, 1, 2), (16, 4, 2, 4), (12, 3, 1, 3)])
def test_select_f64_brute_force(E, G, g_top, k):
    """The exact-mode (fp64, textbook sigmoid) selection used by the finite-difference
    pins, against an exhaustive dominance search over expert and group subsets, with the
    scores and gates checked against their definitions element by element."""
    rng = np.random.default_rng(E + G)
    lg = rng.normal(0, 2, (120, E))
    lg[:10, 1] = lg[:10, 2]                           # exact score ties
    b = rng.normal(0, 0.1, E)
    b[1] = b[2]
    idx, w, s = R.select_f64(lg, b, k, G, g_top)
    for t in range(120):
        v = np.array([1.0 / (1.0 + math.exp(-lg[t, e])) + b[e] for e in range(E)])
        assert list(idx[t]) == _brute_select_f64(v, k, G, g_top), t
        ssel = [1.0 / (1.0 + math.exp(-lg[t, e])) for e in idx[t]]
        assert np.allclose(s[t], ssel, rtol=1e-15, atol=0)
        assert np.allclose(w[t], np.array(ssel) / math.fsum(ssel), rtol=1e-15, atol=0)
