"""Full-prompt cumulated attention (MiniKV's A_cumul) -- oracle (test
infrastructure only).

Follows MiniKV: Pushing the Limits of LLM Inference via 2-Bit Layer-Discriminative
KV Cache, §4.3 "selective flash-attention" and Figure 9, and Algorithm 1 (prefill:
heavy hitters chosen from A_cumul). Every prompt query attends causally to the
prompt keys in the FlashAttention order: the rows are cut into row blocks and,
within a row block, the keys into blocks of KBlockN that are visited one after
another from the first key on; each visit updates every row's running maximum
and forms the tile P = exp(S - running max). The tile is added, column by
column, into A_cumul, and the rows are never normalised (the page leaves the
normalisation out because it would need the whole row first).

So, with S_ij = q_i . k_j / sqrt(d) and j <= i,

    A_cumul[j] = sum over rows i >= j of exp(S_ij - m_i(t(j))),

where t(j) is j's key block and m_i(t) is the maximum of row i's logits over the
key blocks 0..t (keys <= i only).

Readings taken where the page is silent:
  * KBlockN = 128 keys (the page gives tile sizes of 32 to 128 rows; the key
    block is not given). The row block size does not change the result.
  * GQA: the g query heads that share a kv head add their A_cumul into one score
    per kv head, as for the observation-window score.
  * Selection: the last alpha prompt positions stay in the window as for every
    selection, the scores of positions [0, n - alpha) go through the same
    pooling (width 1 leaves them unchanged; MiniKV itself does not pool) and the
    same top-k as the observation-window score.
"""
from __future__ import annotations

import math

import numpy as np

from .snapkv import max_pool, select_topk

KEY_BLOCK = 128


def acumul_scores(q_group: np.ndarray, k: np.ndarray, key_block: int = KEY_BLOCK) -> np.ndarray:
    """A_cumul of one kv head.

    q_group: [g][n][d] -- the queries of every prompt position for the g query
             heads that share this kv head (float64).
    k:       [n][d] keys of this kv head (float64).
    Returns [n]: the column sums of every head's un-normalised tiles, added over
    the g heads.
    """
    q_group = np.asarray(q_group, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    g, n, d = q_group.shape
    if k.shape != (n, d):
        raise ValueError("q_group and k disagree on n or d")
    if key_block < 1:
        raise ValueError("key_block must be positive")
    scale = 1.0 / math.sqrt(d)
    rows = np.arange(n)
    out = np.zeros(n)
    for h in range(g):
        s = (q_group[h] @ k.T) * scale                  # [row][key]
        m = np.full(n, -np.inf)                         # running row maxima
        for t0 in range(0, n, key_block):
            cols = np.arange(t0, min(t0 + key_block, n))
            live = rows >= t0                           # rows that see a key of this block
            tile = s[np.ix_(live, cols)]
            visible = cols[None, :] <= rows[live][:, None]
            tile = np.where(visible, tile, -np.inf)
            m[live] = np.maximum(m[live], tile.max(axis=1))
            p = np.where(visible, np.exp(tile - m[live][:, None]), 0.0)
            out[cols] += p.sum(axis=0)
    return out


def acumul_select(q_group: np.ndarray, k: np.ndarray, budget: int, obs_window: int,
                  pool_kernel: int = 1, key_block: int = KEY_BLOCK):
    """Heavy hitters from A_cumul: the `budget` largest (pooled) scores among
    positions [0, n - obs_window), ties to the lower index, ascending.
    Returns (kept indices, scores, pooled scores)."""
    n = k.shape[0]
    s = acumul_scores(q_group, k, key_block)[:n - obs_window]
    p = max_pool(s, pool_kernel)
    return select_topk(p, budget), s, p


def acumul_columns(q_group: np.ndarray, k: np.ndarray, cols, key_block: int = KEY_BLOCK):
    """A_cumul at the given columns only, each straight from its definition:
    A[j] = sum over rows i >= j of exp(S_ij - m_i), m_i the maximum of row i's
    logits over keys <= i in the key blocks up to and including j's. Cheap for
    columns near either end of a long prompt (few rows, or keys of few blocks)."""
    q_group = np.asarray(q_group, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    g, n, d = q_group.shape
    scale = 1.0 / math.sqrt(d)
    out = []
    for j in cols:
        j = int(j)
        end = min((j // key_block + 1) * key_block, n)   # keys of blocks 0..t(j)
        total = 0.0
        for h in range(g):
            rows = q_group[h, j:]                          # rows i >= j
            s = (rows @ k[:end].T) * scale                 # [i - j][key]
            i = np.arange(j, n)
            s = np.where(np.arange(end)[None, :] <= i[:, None], s, -np.inf)
            m = s.max(axis=1)
            total += float(np.exp(s[:, j] - m).sum())
        out.append(total)
    return np.array(out)


def prefill_attention(q_group: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """X_O of one kv head: the causal softmax attention output of every prompt query
    (MiniKV §4.3, Figure 9: the selective flash-attention kernel returns it beside
    A_cumul). Each row is normalised over its own visible keys:

        X_O[h, i] = sum over j <= i of softmax_j(q_hi . k_j / sqrt(d)) v_j.

    q_group: [g][n][d], k and v: [n][d] (float64). Returns [g][n][d]."""
    q_group = np.asarray(q_group, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    g, n, d = q_group.shape
    scale = 1.0 / math.sqrt(d)
    out = np.empty((g, n, d))
    visible = np.tril(np.ones((n, n), dtype=bool))
    for h in range(g):
        s = np.where(visible, (q_group[h] @ k.T) * scale, -np.inf)
        w = np.exp(s - s.max(axis=1, keepdims=True))
        out[h] = (w / w.sum(axis=1, keepdims=True)) @ v
    return out
