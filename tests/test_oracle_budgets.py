"""Pins the oracle's per-layer budget planner (PyramidKV §4.2 / MiniKV §4.2)."""
import pytest

from oracle import plan_budgets


@pytest.mark.parametrize("L,avg,depth", [(32, 512, 8), (32, 1024, 8), (40, 256, 7),
                                         (7, 96, 3), (2, 64, 2), (1, 128, 8), (33, 2048, 20)])
def test_pyramid_sums_and_shape(L, avg, depth):
    G = 32
    k = plan_budgets(L, "pyramid", avg, depth, G)
    assert len(k) == L
    assert sum(k) == L * avg                        # same total as uniform
    assert all(b % G == 0 and b > 0 for b in k)     # whole quantization groups
    assert all(k[i] >= k[i + 1] for i in range(L - 1))   # lower layers get more
    if L > 1:
        x_u = avg // G
        assert k[-1] == (x_u // depth) * G          # top: x/d
        assert k[0] == (2 * x_u - x_u // depth) * G  # bottom: 2x - x/d


def test_long_context_endpoints():
    """Average 1024, depth 8 over 32 layers: bottom 1920, top 128."""
    k = plan_budgets(32, "pyramid", 1024, 8, 32)
    assert (k[0], k[-1], sum(k)) == (1920, 128, 32 * 1024)


def test_llama3_endpoints():
    k = plan_budgets(32, "pyramid", 512, 8, 32)
    assert (k[0], k[-1], sum(k)) == (960, 64, 16_384)


def test_pyramid_is_linear_within_one_group():
    """Each budget is within one group of the exact arithmetic sequence."""
    L, avg, d, G = 32, 512, 8, 32
    k = plan_budgets(L, "pyramid", avg, d, G)
    top, bottom = (avg // G // d) * G, (2 * (avg // G) - avg // G // d) * G
    for l, b in enumerate(k):
        exact = bottom - (bottom - top) * l / (L - 1)
        assert abs(b - exact) < G


def test_uniform_and_clip():
    assert plan_budgets(4, "uniform", 128, 0, 32) == [128] * 4
    assert max(plan_budgets(3, "pyramid", 512, 8, 32, max_budget=300)) <= 300
    assert plan_budgets(5, "none", 0, 0, 32, max_budget=777) == [777] * 5


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        plan_budgets(4, "uniform", 100, 0, 32)      # not whole groups
    with pytest.raises(ValueError):
        plan_budgets(4, "pyramid", 128, 0, 32)
    with pytest.raises(ValueError):
        plan_budgets(4, "bogus", 128, 2, 32)
