"""Pins the oracle's variance score and variance-driven budget planner (MiniKV
§4.2 "Layer-Specific Selectivity", Var-prop / Var-inv; Figure 7's variance score)."""
import itertools
from fractions import Fraction

import numpy as np
import pytest

from oracle import plan_budgets
from oracle.variance import (integer_weights, layer_variance, plan_budgets_weighted,
                             score_variance, variance_weights)


# ------------------------------------------------------------------ variance score
@pytest.mark.parametrize("m", [1, 2, 7, 100, 4097])
def test_variance_of_arithmetic_sequence(m):
    """0, 1, ..., m-1 has population variance (m^2 - 1) / 12."""
    assert score_variance(np.arange(m)) == pytest.approx((m * m - 1) / 12, rel=1e-13, abs=1e-13)


def test_variance_shift_scale_and_constant():
    rng = np.random.default_rng(3)
    s = rng.exponential(size=999)
    v = score_variance(s)
    assert score_variance(s + 17.0) == pytest.approx(v, rel=1e-11)     # shift-invariant
    assert score_variance(3.0 * s) == pytest.approx(9.0 * v, rel=1e-13)  # scales by c^2
    assert score_variance(np.full(50, 2.5)) == 0.0


def test_variance_of_two_point_distribution():
    """k ones among m values: variance p (1 - p), p = k / m (Bernoulli)."""
    m, k = 64, 5
    s = np.zeros(m)
    s[:k] = 1.0
    p = k / m
    assert score_variance(s) == pytest.approx(p * (1 - p), rel=1e-14)


def test_layer_variance_is_mean_over_units():
    sc = np.zeros((2, 3, 10))
    sc[0, 0, 0] = 10.0          # variance 10^2 * (1/10)(9/10) = 9
    sc[1, 2] = np.arange(10)    # variance 99 / 12
    assert layer_variance(sc) == pytest.approx((9.0 + 99 / 12) / 6, rel=1e-14)


# ------------------------------------------------------------------ the planner
def test_equal_weights_give_the_uniform_schedule():
    for L, avg in [(32, 512), (7, 96), (1, 64), (40, 128)]:
        assert plan_budgets_weighted(L, avg, [2.5] * L, 32) == plan_budgets(L, "uniform", avg,
                                                                            0, 32)


@pytest.mark.parametrize("L,avg,seed", [(32, 512, 0), (32, 1024, 1), (7, 96, 2), (3, 64, 3),
                                        (40, 256, 4), (5, 32, 5)])
def test_sum_groups_and_proportionality(L, avg, seed):
    G = 32
    w = list(np.random.default_rng(seed).lognormal(0.0, 1.0, L))
    k = plan_budgets_weighted(L, avg, w, G)
    assert sum(k) == L * avg
    assert all(b % G == 0 and b >= G for b in k)
    q = integer_weights(w)
    spare = L * (avg // G) - L
    for l in range(L):
        quota = Fraction(spare * q[l], sum(q))
        assert abs(Fraction(k[l] // G - 1) - quota) < 1     # floor or ceil of its quota


def test_largest_remainder_minimises_squared_deviation():
    """Brute force on tiny cases: among all ways to share the spare groups, the
    plan is the one closest to the exact quotas in squared deviation (the
    Hamilton apportionment's defining property); ties to the lower layers."""
    G = 32
    rng = np.random.default_rng(11)
    for _ in range(40):
        L = int(rng.integers(1, 5))
        avg_u = int(rng.integers(1, 6))
        w = [float(x) for x in rng.integers(1, 9, L)]
        got = [b // G - 1 for b in plan_budgets_weighted(L, avg_u * G, w, G)]
        q = integer_weights(w)
        spare = L * avg_u - L
        quota = [Fraction(spare * ql, sum(q)) for ql in q]
        best = None
        for u in itertools.product(range(spare + 1), repeat=L):
            if sum(u) != spare:
                continue
            dev = sum((Fraction(ui) - qi) ** 2 for ui, qi in zip(u, quota))
            key = (dev, [-x for x in u])        # prefer more groups in lower layers
            if best is None or key < best[0]:
                best = (key, list(u))
        assert got == best[1], (w, avg_u, got, best[1])


def test_var_prop_and_var_inv_orientation():
    var = [4.0, 2.0, 1.0, 0.5]
    prop = plan_budgets_weighted(4, 256, variance_weights(var, "var-prop"), 32)
    inv = plan_budgets_weighted(4, 256, variance_weights(var, "var-inv"), 32)
    assert prop == sorted(prop, reverse=True) and prop[0] > prop[-1]
    assert inv == sorted(inv) and inv[0] < inv[-1]
    assert prop == inv[::-1]                       # mirrored weights, mirrored plan
    # exact shares: spare 28 groups in proportion 8:4:2:1 -> 14.93, 7.47, 3.73, 1.87
    assert prop == [(1 + u) * 32 for u in (15, 7, 4, 2)]


def test_scale_invariance_and_clip():
    w = [0.3, 1.7, 0.9, 2.2, 0.05]
    k = plan_budgets_weighted(5, 160, w, 32)
    assert plan_budgets_weighted(5, 160, [4.0 * x for x in w], 32) == k
    assert max(plan_budgets_weighted(5, 160, w, 32, max_budget=200)) <= 200


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        plan_budgets_weighted(3, 64, [1.0, 0.0, 1.0], 32)
    with pytest.raises(ValueError):
        plan_budgets_weighted(3, 64, [1.0, float("inf"), 1.0], 32)
    with pytest.raises(ValueError):
        plan_budgets_weighted(3, 48, [1.0, 1.0, 1.0], 32)
    with pytest.raises(ValueError):
        plan_budgets_weighted(3, 64, [1.0, 1.0], 32)
    with pytest.raises(ValueError):
        variance_weights([1.0, 0.0], "var-inv")
