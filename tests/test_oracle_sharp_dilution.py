"""The attention-mass dilution diagnostic (oracle/sharp_dilution.py) against
what mathematics fixes: brute force over subsets, closed forms, invariances,
and the direction of the effect the SharpDraft abstract describes."""
import itertools
import math

import numpy as np
import pytest

from oracle import sharp_dilution as sd


def test_equal_logits_give_k_over_n():
    for n, k in [(1, 1), (10, 3), (4096, 8)]:
        assert sd.topk_mass(np.full(n, 1.7), k) == pytest.approx(k / n, rel=1e-12)


def test_brute_force_over_subsets():
    rng = np.random.default_rng(3)
    for _ in range(20):
        s = rng.normal(0, 2, size=6)
        p = np.exp(s) / np.exp(s).sum()
        for k in range(1, 7):
            best = max(sum(p[list(c)]) for c in itertools.combinations(range(6), k))
            assert sd.topk_mass(s, k) == pytest.approx(best, rel=1e-12)


def test_shift_invariance_and_edges():
    s = np.random.default_rng(5).normal(size=100)
    assert sd.topk_mass(s + 123.0, 7) == pytest.approx(sd.topk_mass(s, 7), rel=1e-12)
    assert sd.topk_mass(s, 100) == pytest.approx(1.0, rel=1e-12)
    assert sd.topk_mass(s, 500) == pytest.approx(1.0, rel=1e-12)
    assert sd.topk_mass(s, 0) == 0.0


def test_two_level_closed_form():
    # k keys at logit a, n - k at 0: mass = k e^a / (k e^a + n - k)
    for n, k, a in [(1000, 4, 3.0), (65536, 8, 6.0), (50, 50, 1.0)]:
        s = np.zeros(n)
        s[:k] = a
        want = k * math.exp(a) / (k * math.exp(a) + n - k)
        assert sd.topk_mass(s, k) == pytest.approx(want, rel=1e-12)


def test_dilution_and_query_scaling():
    ns = [4096, 65536, 1 << 20]
    rows = sd.dilution_curve(ns, draws=4)
    plain = [r["topk_mass"] for r in rows]
    sharp = [r["topk_mass_sharp"] for r in rows]
    assert plain[0] > plain[1] > plain[2]                       # mass dilutes as n grows
    assert rows[0]["gamma"] == 1.0 and sharp[0] == pytest.approx(plain[0], rel=1e-12)
    assert all(s_ > p_ for s_, p_ in zip(sharp[1:], plain[1:]))  # the scale restores some mass
    flat = sd.dilution_curve(ns, beta=0.0, draws=2, seed=9)
    assert all(r["gamma"] == 1.0 and r["topk_mass"] == r["topk_mass_sharp"] for r in flat)


def test_relevant_keys_are_the_top_k():
    rng = np.random.default_rng(1)
    s = sd.synthetic_logits(1 << 16, 8, 6.0, 1.0, rng)
    assert set(np.argsort(s)[-8:]) == set(range(8))
