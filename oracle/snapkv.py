"""Observation-window scoring, pooling and per-head top-k -- oracle (test only).

Follows:
  * PyramidKV: Dynamic KV Cache Compression based on Pyramidal Information
    Funneling, §4.2.2 "KV Cache Selection": the last alpha prompt tokens (the
    "instruction tokens") are always kept; every other token i gets the score
    s_i^h = the attention the instruction tokens pay it in head h, a pooling layer
    smooths the scores so massive activations do not mislead the selection, and
    the top k^l tokens per head are kept, the rest discarded for good.
  * MiniKV: Pushing the Limits of LLM Inference via 2-Bit Layer-Discriminative KV
    Cache, §2 eq. (1): A = softmax(Q K^T / sqrt(d)).
  * KV Cache Compression: Eviction and Quantization (blog), "Eviction: keep fewer
    tokens": SnapKV looks at the attention the prompt's last tokens pay the rest,
    per head, and keeps the positions they attend to.

Readings (the score and pooling equations are lost on the PyramidKV page):
  * Attention is causal (prefill is causal): instruction token j sees keys 0..j.
  * Softmax rows are normalised (A is a true softmax), then summed over the
    window's rows and over all query heads of a GQA group (the pages are silent on
    GQA; summing the group gives one score per kv head, which is what is evicted).
  * Pooling is a stride-1 max over [i - (w-1)/2, i + (w-1)/2] clipped to the
    scored range [0, n - alpha), applied after the window/group sum.
  * Top-k ties go to the lower index; the kept indices are returned ascending.

Parity unpinned as to the reading: no page prints a worked selection, so the
order of the GQA sum and the pool (sum first, then pool) is a reading, not a
pinned fact. The arithmetic of that reading is pinned (closed forms, brute force,
scipy's maximum filter).
"""
from __future__ import annotations

import math

import numpy as np


def window_scores(q_group: np.ndarray, k: np.ndarray) -> np.ndarray:
    """Column sums of the causal softmax attention of the observation rows.

    q_group: [g][alpha][d] -- queries of the last alpha prompt positions for the g
             query heads that share this kv head (float64).
    k:       [n][d] keys of this kv head (float64).
    Returns col [n] with col[i] = sum over heads and rows j of A[j, i]; the
    selection scores are col[:n - alpha]. Each softmax row sums to one, so
    col.sum() == g * alpha.
    """
    g, a, d = q_group.shape
    n = k.shape[0]
    rows = q_group.reshape(g * a, d).astype(np.float64)
    pos = np.tile(np.arange(n - a, n), g)                       # prompt position of each row
    logits = (rows @ k.astype(np.float64).T) / math.sqrt(d)     # [g*a][n]
    logits[np.arange(n)[None, :] > pos[:, None]] = -np.inf       # causal
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    attn = e / e.sum(axis=1, keepdims=True)
    return attn.sum(axis=0)


def max_pool(s: np.ndarray, w: int) -> np.ndarray:
    """Stride-1 1-D max-pool of width w (odd), window clipped to the array."""
    if w < 1 or w % 2 == 0:
        raise ValueError("pool kernel must be odd and >= 1")
    r = (w - 1) // 2
    padded = np.pad(np.asarray(s, dtype=np.float64), r, constant_values=-np.inf)
    return np.lib.stride_tricks.sliding_window_view(padded, w).max(axis=1)


def select_topk(p: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries of p, ties to the lower index, ascending."""
    n = len(p)
    if k >= n:
        return np.arange(n, dtype=np.int64)
    order = np.argsort(-np.asarray(p, dtype=np.float64), kind="stable")
    return np.sort(order[:k]).astype(np.int64)


def snapkv_select(q_group: np.ndarray, k: np.ndarray, budget: int, pool_kernel: int):
    """Full selection for one (sequence, kv head).

    Returns (kept indices ascending, scores s[:n-alpha], pooled p[:n-alpha]).
    """
    a = q_group.shape[1]
    n = k.shape[0]
    col = window_scores(q_group, k)
    s = col[: n - a]
    p = max_pool(s, pool_kernel)
    return select_topk(p, budget), s, p
