"""Pins of the sink + recent-window selection (oracle/sinks.py) against what the
pages fix: the blog's '4 sink tokens + the last 508' within a budget of 512, the
PyramidKV baseline's 'first k - alpha and last alpha' (every kept position a
prefix one when n_sinks = k), and brute-force enumeration of the definition."""
import numpy as np
import pytest

from oracle import sinks_window_select


def test_blog_budget_512_four_sinks():
    n = 2048 - 16                      # scored range before a 16-token window
    kept = sinks_window_select(n, 512, 4)
    assert len(kept) == 512
    assert list(kept[:4]) == [0, 1, 2, 3]
    assert list(kept[4:]) == list(range(n - 508, n))


def test_no_sinks_is_pure_recency():
    assert list(sinks_window_select(100, 10, 0)) == list(range(90, 100))


def test_all_sinks_is_the_prefix():
    # PyramidKV's StreamingLLM baseline: the first k - alpha positions (the last
    # alpha are the observation window, kept separately)
    assert list(sinks_window_select(100, 10, 10)) == list(range(10))
    assert list(sinks_window_select(100, 10, 50)) == list(range(10))


def test_budget_at_least_the_range_keeps_everything():
    assert list(sinks_window_select(37, 37, 4)) == list(range(37))
    assert list(sinks_window_select(37, 1000, 4)) == list(range(37))


def test_brute_force_definition():
    for n in range(0, 12):
        for k in range(0, 14):
            for s in range(0, 6):
                kept = sinks_window_select(n, k, s)
                kk = min(k, n)
                ss = min(s, kk)
                ref = sorted(set(range(ss)) | set(range(n - (kk - ss), n))) if kk < n \
                    else list(range(n))
                assert list(kept) == ref, (n, k, s)
                assert len(kept) == kk
                assert np.all(np.diff(kept) > 0)


def test_rejects_negative_sizes():
    with pytest.raises(ValueError):
        sinks_window_select(10, 5, -1)
