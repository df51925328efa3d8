"""Variance-driven per-layer budgets (Var-prop / Var-inv) -- oracle (test
infrastructure only).

Follows MiniKV: Pushing the Limits of LLM Inference via 2-Bit Layer-Discriminative
KV Cache, §4.2 "Layer-Specific Selectivity" (the "Variance" policy) and Figure 7:
a layer's variance score is the variance of its cumulated attention; Var-prop
gives each layer a cache budget proportional to that variance, Var-inv one
inversely proportional to it, at the same average budget.

Readings taken where the page is silent:
  * A layer's cumulated attention is the selection score this path computes
    (observation-window softmax rows summed over the window and the GQA group,
    before pooling): one vector per (sequence, kv head) over the n - alpha
    selectable positions. Its variance is the population variance over those
    positions; the layer's variance score is the mean of it over the
    (sequence, kv head) units. (MiniKV's own score is the full-prompt column sum
    without row normalisation; this path's scores are the ones it has.)
  * The page observes that the variance profile of a model hardly changes across
    datasets, so the scores come from a profiling prefill and the budgets are
    planned before the cache is created.
  * Budgets are whole quantization groups of G tokens and every layer keeps at
    least one group. The remaining L*x/G - L groups are shared in proportion to
    the weights by the largest-remainder rule: each quota is floored and the
    leftover groups go one each to the largest remainders, ties to the lower
    layer, so the budgets sum to exactly L*x as for the other schedules.
  * For exact integer shares every weight is first scaled to an integer,
    q_l = max(1, rint(w_l / max(w) * 2^30)) (IEEE double division, round half to
    even); the quota of layer l is (spare * q_l) / sum(q) in exact integers.
  * Budgets are finally clipped to the selectable prompt tokens, as for the other
    schedules.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence

import numpy as np

WEIGHT_SCALE = 2 ** 30


def score_variance(s) -> float:
    """Population variance of one (sequence, kv head)'s scores s_0..s_{m-1}:
    mean of (s_i - mean(s))^2, in fp64."""
    s = np.asarray(s, dtype=np.float64)
    if s.size == 0:
        raise ValueError("no scores")
    mu = s.sum() / s.size
    return float(((s - mu) ** 2).sum() / s.size)


def layer_variance(scores) -> float:
    """A layer's variance score: the mean over (sequence, kv head) units of the
    per-unit score variance. scores: [B][H][m]."""
    sc = np.asarray(scores, dtype=np.float64)
    per_unit = [score_variance(sc[b, h]) for b in range(sc.shape[0]) for h in range(sc.shape[1])]
    return float(sum(per_unit) / len(per_unit))


def variance_weights(variances: Sequence[float], policy: str) -> List[float]:
    """Per-layer weights of a variance policy: "var-prop" (w = variance) or
    "var-inv" (w = 1 / variance)."""
    v = [float(x) for x in variances]
    if any(not math.isfinite(x) or x <= 0 for x in v):
        raise ValueError("variances must be positive and finite")
    if policy == "var-prop":
        return v
    if policy == "var-inv":
        return [1.0 / x for x in v]
    raise ValueError(f"unknown policy {policy!r}")


def integer_weights(weights: Sequence[float]) -> List[int]:
    """q_l = max(1, rint(w_l / max(w) * 2^30))."""
    w = [float(x) for x in weights]
    if not w or any(not math.isfinite(x) or x <= 0 for x in w):
        raise ValueError("weights must be positive and finite")
    wmax = max(w)
    return [max(1, int(np.rint((x / wmax) * WEIGHT_SCALE))) for x in w]


def plan_budgets_weighted(n_layers: int, avg_budget: int, weights: Sequence[float],
                          group_size: int, max_budget: Optional[int] = None) -> List[int]:
    """Per-layer budgets (tokens) proportional to `weights`, one group at least each."""
    L, G = int(n_layers), int(group_size)
    if L <= 0 or G <= 0 or len(weights) != L:
        raise ValueError("need one weight per layer")
    if avg_budget <= 0 or avg_budget % G:
        raise ValueError("avg_budget must be a positive multiple of group_size")
    q = integer_weights(weights)
    total = L * (avg_budget // G)
    spare = total - L                      # after the one group every layer keeps
    qsum = sum(q)
    units = [1 + spare * ql // qsum for ql in q]
    rem = [spare * ql % qsum for ql in q]
    left = total - sum(units)
    for l in sorted(range(L), key=lambda l: (-rem[l], l))[:left]:
        units[l] += 1
    budgets = [u * G for u in units]
    if max_budget is not None:
        budgets = [min(b, int(max_budget)) for b in budgets]
    return budgets
