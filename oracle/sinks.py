"""Attention-sink + recent-token selection -- oracle (test infrastructure only).

Follows:
  * KV Cache Compression: Eviction and Quantization (blog), "Measured on a real
    model" and "Attention sinks": keeping only the most recent tokens loses the
    first few tokens that every query parks attention on; the policy that works
    keeps the first 4 tokens plus the most recent ones within the same budget
    (the table's "4 sink tokens + the last 508" against "the last 512").
  * PyramidKV: Dynamic KV Cache Compression based on Pyramidal Information
    Funneling, related work / baselines (StreamingLLM): its StreamingLLM baseline
    keeps the last alpha tokens and the first k - alpha ones.

Reading: per (sequence, kv head), of the scored range [0, n - alpha) (the last
alpha prompt tokens are kept in the window as with every selection) the budget k
keeps the first s = min(n_sinks, k) positions and the k - s positions just before
the observation window; with n_sinks = k this is PyramidKV's baseline, with
n_sinks = 4 the blog's. k >= n - alpha keeps everything. Indices ascending.
"""
from __future__ import annotations

import numpy as np


def sinks_window_select(n_scored: int, budget: int, n_sinks: int) -> np.ndarray:
    """Kept positions (ascending int64) of the sink + recent-window policy."""
    if n_scored < 0 or budget < 0 or n_sinks < 0:
        raise ValueError("sizes must be non-negative")
    k = min(budget, n_scored)
    if k == n_scored:
        return np.arange(n_scored, dtype=np.int64)
    s = min(n_sinks, k)
    recent = np.arange(n_scored - (k - s), n_scored, dtype=np.int64)
    return np.concatenate([np.arange(s, dtype=np.int64), recent])
