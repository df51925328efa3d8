"""Pins the oracle's observation-window scoring, pooling and top-k."""
import itertools
import math

import numpy as np
import pytest
from scipy.ndimage import maximum_filter1d

from oracle import window_scores, max_pool, select_topk, snapkv_select


def test_uniform_attention_closed_form():
    """Identical keys: causal row j attends 1/(j+1) to each key 0..j (harmonic sums)."""
    rng = np.random.default_rng(0)
    g, a, d, n = 3, 5, 16, 40
    k = np.tile(rng.normal(size=d), (n, 1))
    q = rng.normal(size=(g, a, d))
    col = window_scores(q, k)
    harmonic = sum(1.0 / (j + 1) for j in range(n - a, n))
    np.testing.assert_allclose(col[: n - a], g * harmonic, rtol=1e-13)
    # key i inside the window is seen only by rows j >= i
    for i in range(n - a, n):
        np.testing.assert_allclose(col[i], g * sum(1.0 / (j + 1) for j in range(i, n)),
                                   rtol=1e-13)


def test_rows_sum_to_one():
    rng = np.random.default_rng(1)
    g, a, d, n = 4, 8, 32, 300
    col = window_scores(rng.normal(size=(g, a, d)) * 2, rng.normal(size=(n, d)))
    assert abs(col.sum() - g * a) < 1e-10
    assert (col >= 0).all()


def test_two_keys_scale_and_diagonal():
    """n = 2, one observation row (position 1): score of key 0 is a logistic in
    (l0 - l1) / sqrt(d) -- pins the 1/sqrt(d) scale and that the row sees itself."""
    d = 64
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 3.0
    k = np.zeros((2, d)); k[0, 0] = 2.0; k[1, 0] = -1.0
    l0, l1 = 6.0, -3.0
    s0 = window_scores(q, k)[0]
    assert s0 == pytest.approx(1.0 / (1.0 + math.exp((l1 - l0) / math.sqrt(d))), rel=1e-14)


def test_gqa_heads_are_summed():
    rng = np.random.default_rng(2)
    a, d, n = 4, 8, 50
    k = rng.normal(size=(n, d))
    q = rng.normal(size=(2, a, d))
    both = window_scores(q, k)
    np.testing.assert_allclose(both, window_scores(q[:1], k) + window_scores(q[1:], k),
                               rtol=1e-13)


def test_pool_matches_library_filter():
    rng = np.random.default_rng(3)
    for w in (1, 3, 7, 9):
        s = rng.random(97)
        np.testing.assert_array_equal(max_pool(s, w),
                                      maximum_filter1d(s, size=w, mode="nearest"))
    # windows as wide as or wider than the row (short prompts): every position
    # sees the whole row, or all of it within reach
    for n, w in ((1, 7), (3, 7), (5, 11), (6, 7), (7, 25)):
        s = rng.random(n)
        np.testing.assert_array_equal(max_pool(s, w),
                                      maximum_filter1d(s, size=w, mode="nearest"))
    np.testing.assert_array_equal(max_pool(np.array([0.2, 0.9, 0.1]), 25), [0.9, 0.9, 0.9])


def test_pool_rejects_even_kernel():
    with pytest.raises(ValueError):
        max_pool(np.zeros(5), 4)


def _brute_topk(p, k):
    """i is kept iff fewer than k entries beat it (larger value, or equal at a lower index)."""
    n = len(p)
    keep = [i for i in range(n)
            if sum(1 for j in range(n) if p[j] > p[i] or (p[j] == p[i] and j < i)) < k]
    return np.array(sorted(keep), dtype=np.int64)


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(4)
    for trial in range(300):
        n = int(rng.integers(1, 12))
        p = rng.integers(0, 4, size=n).astype(float)     # many exact ties
        k = int(rng.integers(0, n + 2))
        np.testing.assert_array_equal(select_topk(p, k), _brute_topk(p, k))


def test_topk_enumeration_tiny():
    """Over all subsets of size k: the kept set has the largest sum, and among the
    maximal ones the lexicographically smallest index tuple."""
    rng = np.random.default_rng(5)
    for trial in range(50):
        n = int(rng.integers(2, 8))
        p = rng.integers(0, 3, size=n).astype(float)
        k = int(rng.integers(1, n))
        best = max(itertools.combinations(range(n), k),
                   key=lambda c: (sum(p[i] for i in c), [-i for i in c]))
        np.testing.assert_array_equal(select_topk(p, k), np.array(best))


def test_planted_sinks_and_needles_are_kept():
    """Keys aligned with the queries (x4 norm) dominate the window's attention."""
    import synth
    spec = synth.small_spec(5, n_layers=1, prompt_len=2048, obs_window=64, avg_budget=128,
                            needles=16)
    x = synth.layer_inputs(spec, 0)
    k = x["k"].double().numpy()
    q = x["q_obs"].double().numpy()
    g = spec.gqa
    for h in range(spec.n_kv_heads):
        kept, s, p = snapkv_select(q[0, h * g:(h + 1) * g], k[0, h], 128, 7)
        needles = set(x["needles"][0, h].tolist())
        assert needles <= set(kept.tolist())
        assert set(x["sinks"]) <= set(kept.tolist())
