"""Per-layer token budgets k^l -- oracle (test infrastructure only).

Follows:
  * PyramidKV: Dynamic KV Cache Compression based on Pyramidal Information
    Funneling, §4.2 "Proposed Method" (budget allocation): lower layers get more
    cache than upper layers, the bottom and top budgets are fixed first and the
    layers in between follow an arithmetic sequence (the sequence's equation is
    lost on the page).
  * MiniKV: Pushing the Limits of LLM Inference via 2-Bit Layer-Discriminative KV
    Cache, §4.2 "Layer-Specific Selectivity" (Pyramid): for an average budget x and
    pyramid depth d the two end layers get x/d and 2x - x/d, linear in between, so
    the budgets sum to exactly (number of layers) * x; "Uniform": every layer x.

Readings taken where the pages are silent or disagree:
  * Orientation: more budget at the bottom (layer 0 gets 2x - x/d, the top layer
    x/d), as both pages say in words; MiniKV's sentence that gives x/d to the
    bottom-most layer contradicts its own "more cache in lower layers".
  * PyramidKV's endpoints 2k/m and k/(beta m) do not sum to k for a linear
    sequence (they overshoot by k/(2 beta)); MiniKV's endpoints do, so they are used.
  * The sequence is taken in whole quantization groups (units of G tokens, so the
    packed store holds whole groups): unit budget
      r_l = (B_u (L-1) - (B_u - T_u) l) / (L-1),  T_u = floor(x_u / d), B_u = 2 x_u - T_u,
    x_u = x / G. Each r_l is floored, and the units left over (the sum of the
    fractional parts, an integer) go one each to the layers with the largest
    remainders, ties to the lower layer. All integer arithmetic.
  * Budgets are finally clipped to the number of selectable prompt tokens.

Parity unpinned as to the reading: which endpoints the pages mean (MiniKV's x/d
form rather than PyramidKV's beta form) is a reading, not a pinned fact. The
schedule it gives is pinned (exact sums, the long-context workload's 1,920 / 128
endpoints, one group from the exact line).
"""
from __future__ import annotations

from typing import List, Optional


def plan_budgets(n_layers: int, schedule: str, avg_budget: int, pyramid_depth: int,
                 group_size: int, max_budget: Optional[int] = None) -> List[int]:
    """Return the per-layer budgets (tokens) k^0..k^{L-1}.

    schedule: "uniform" | "pyramid" | "none" ("none" keeps every token: the
    budget is `max_budget`).
    """
    L, G = int(n_layers), int(group_size)
    if L <= 0 or G <= 0:
        raise ValueError("n_layers and group_size must be positive")
    if schedule == "none":
        if max_budget is None:
            raise ValueError("schedule 'none' needs max_budget")
        return [int(max_budget)] * L
    if avg_budget <= 0 or avg_budget % G:
        raise ValueError("avg_budget must be a positive multiple of group_size")
    x_u = avg_budget // G
    if schedule == "uniform":
        units = [x_u] * L
    elif schedule == "pyramid":
        if pyramid_depth < 1:
            raise ValueError("pyramid_depth must be >= 1")
        top = x_u // pyramid_depth
        bottom = 2 * x_u - top
        total = L * x_u
        if L == 1:
            units = [x_u]
        else:
            den = L - 1
            num = [bottom * den - (bottom - top) * l for l in range(L)]
            units = [v // den for v in num]
            rem = [v % den for v in num]
            left = total - sum(units)
            order = sorted(range(L), key=lambda l: (-rem[l], l))
            for l in order[:left]:
                units[l] += 1
    else:
        raise ValueError(f"unknown schedule {schedule!r}")
    budgets = [u * G for u in units]
    if max_budget is not None:
        budgets = [min(b, int(max_budget)) for b in budgets]
    return budgets
