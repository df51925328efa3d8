"""Variance-driven budgets on the GPU (MiniKV §4.2 "Layer-Specific Selectivity",
Var-prop / Var-inv; Figure 7's variance score): the per-(sequence, kv head)
variance of each layer's selection scores against the oracle, budgets planned
from those variances, and a cache built on them against the oracle end to end."""
import numpy as np
import pytest
import torch

import synth
from _parity import DECODE_RTOL, kvc, np64, run_small
from oracle import (OracleCache, acumul_scores, layer_variance, plan_budgets_weighted,
                    score_variance, variance_weights)

pytestmark = pytest.mark.gpu

SPEC = synth.small_spec(2, n_layers=3, batch=2, n_q_heads=8, n_kv_heads=2, prompt_len=1000,
                        obs_window=32, avg_budget=96, schedule="uniform", window_len=64)


def _profile_variances(spec):
    """Profiling prefill (uniform budgets): per layer the GPU's per-unit variances,
    its own scores, and the oracle's scores."""
    K = kvc()
    dims = K.dims_from_spec(spec, max_new_tokens=4)
    budgets = K.kvc_plan_budgets(dims, "uniform", spec.avg_budget)
    B, Hk, g = spec.batch, spec.n_kv_heads, spec.gqa
    ns = spec.prompt_len - spec.obs_window
    cache = None
    out = []
    for layer in range(spec.n_layers):
        x = synth.layer_inputs(spec, layer, device="cuda")
        cache = K.kvc_prefill_compress(dims, budgets, layer, x["q_obs"], x["k"], x["v"],
                                       cache=cache)
        var = torch.empty(B, Hk, device="cuda")
        sc = torch.empty(B, Hk, ns, device="cuda")
        K.kvc_score_variance(cache, var)
        K.kvc_scores_layer(cache, sc)
        torch.cuda.synchronize()
        oc = OracleCache(B, spec.n_q_heads, Hk, spec.head_dim, spec.bits, spec.group_size,
                         spec.window_len)
        oc.prefill(np64(x["k"]), np64(x["v"]), spec.obs_window, budget=budgets[layer],
                   q_obs=np64(x["q_obs"]), pool_kernel=spec.pool_kernel)
        out.append((var.double().cpu().numpy(), sc.double().cpu().numpy(), oc))
    K.kvc_check_device(cache)
    cache.close()
    return out


def test_score_variance_matches_oracle():
    worst_own = worst_ora = 0.0
    for var, sc, oc in _profile_variances(SPEC):
        for b in range(SPEC.batch):
            for h in range(SPEC.n_kv_heads):
                own = score_variance(sc[b, h])             # the GPU's scores, fp64
                ora = score_variance(oc.scores[b][h])      # the oracle's scores
                worst_own = max(worst_own, abs(var[b, h] - own) / own)
                worst_ora = max(worst_ora, abs(var[b, h] - ora) / ora)
    print(f"variance vs own scores {worst_own:.2e}, vs oracle {worst_ora:.2e}")
    # the reduction: the scores cut into slices, one CTA each; each thread's
    # compensated (Kahan) fp32 sums of its elements and of their squared deviations
    # about the slice's fp32-rounded mean (each square rounded once to fp32, 2^-24
    # relative; the mean's rounding corrected in fp64), added across a warp in
    # double-float and across warps in fp64; the slices' (count, sum, M2) merged
    # pairwise in fp64; the result rounded to fp32: a few fp32 ulps in all at these
    # lengths, far below 1e-6
    assert worst_own <= 1e-6
    assert worst_ora <= 1e-3        # plus the scores' own tolerance (1e-4 each)


@pytest.mark.parametrize("policy", ["var-prop", "var-inv"])
def test_variance_budgets_end_to_end(policy):
    """Budgets from the GPU's layer variances (C planner == oracle planner), then
    compression with those budgets and 30 decode steps against the oracle."""
    K = kvc()
    prof = _profile_variances(SPEC)
    layer_var = [float(v.mean()) for v, _, _ in prof]
    w = variance_weights(layer_var, policy)
    dims = K.dims_from_spec(SPEC, max_new_tokens=30)
    avg = 320          # 10 groups a layer: enough spare groups for the shares to differ
    budgets = K.kvc_plan_budgets_weighted(dims, avg, w)
    ns = SPEC.prompt_len - SPEC.obs_window
    assert budgets == plan_budgets_weighted(SPEC.n_layers, avg, w, SPEC.group_size,
                                            max_budget=ns)
    assert sum(budgets) == SPEC.n_layers * avg and len(set(budgets)) > 1
    print(policy, "layer variances", [f"{v:.3g}" for v in layer_var], "budgets", budgets)
    rep = run_small(SPEC, 30, selection="score", budgets=budgets)
    assert rep.decode_checked > 0 and rep.decode_err <= DECODE_RTOL


def test_score_variance_needs_a_scored_layer():
    K = kvc()
    dims = K.dims_from_spec(SPEC, max_new_tokens=4)
    cache = K.kvc_cache_create(dims, K.kvc_plan_budgets(dims, "uniform", SPEC.avg_budget))
    var = torch.empty(SPEC.batch, SPEC.n_kv_heads, device="cuda")
    with pytest.raises(K.KvcError) as e:
        K.kvc_score_variance(cache, var)
    assert e.value.status == 5
    cache.close()


ACUMUL_SPEC = synth.small_spec(2, n_layers=3, batch=1, n_q_heads=8, n_kv_heads=2,
                               prompt_len=800, obs_window=32, avg_budget=96,
                               schedule="uniform", window_len=64)


def test_variance_of_cumulated_attention():
    """MiniKV Figure 7's variance score is that of the cumulated attention: the
    variance after kvc_prefill_acumul against the oracle's A_cumul of the same
    inputs, per unit and per layer; then Var-prop budgets from it, and a cache
    selected by A_cumul under those budgets against the oracle end to end."""
    K = kvc()
    spec = ACUMUL_SPEC
    dims = K.dims_from_spec(spec, max_new_tokens=4)
    budgets = K.kvc_plan_budgets(dims, "uniform", spec.avg_budget)
    B, Hk, g = spec.batch, spec.n_kv_heads, spec.gqa
    ns = spec.prompt_len - spec.obs_window
    cache = K.kvc_cache_create(dims, budgets)
    layer_var, worst = [], 0.0
    for layer in range(spec.n_layers):
        x = synth.layer_inputs(spec, layer, device="cuda")
        qf = synth.prompt_queries(spec, layer, device="cuda")
        K.kvc_prefill_acumul(cache, layer, qf, x["k"], x["v"])
        var = torch.empty(B, Hk, device="cuda")
        K.kvc_score_variance(cache, var)
        torch.cuda.synchronize()
        q_np, k_np = np64(qf), np64(x["k"])
        ora = np.stack([[acumul_scores(q_np[b, h * g:(h + 1) * g], k_np[b, h])[:ns]
                         for h in range(Hk)] for b in range(B)])
        v = var.double().cpu().numpy()
        for b in range(B):
            for h in range(Hk):
                ref = score_variance(ora[b, h])
                worst = max(worst, abs(v[b, h] - ref) / ref)
        layer_var.append(float(v.mean()))
        assert abs(layer_var[-1] - layer_variance(ora)) <= 1e-3 * layer_variance(ora)
    K.kvc_check_device(cache)
    cache.close()
    print(f"Var(A_cumul) vs oracle: worst relative error {worst:.2e}; layers "
          f"{[f'{x:.4g}' for x in layer_var]}")
    assert worst <= 1e-3          # the scores' own tolerance carried into the variance
    w = variance_weights(layer_var, "var-prop")
    avg = 160
    budgets = K.kvc_plan_budgets_weighted(dims, avg, w)
    assert budgets == plan_budgets_weighted(spec.n_layers, avg, w, spec.group_size,
                                            max_budget=ns)
    rep = run_small(spec, 20, selection="acumul", budgets=budgets)
    assert rep.decode_checked > 0 and rep.decode_err <= DECODE_RTOL
