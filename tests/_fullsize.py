"""Parity at the workloads' full sizes, in the launch configuration the benchmark
times: every layer compressed with one kvc_prefill_compress call, every decode
step one kvc_decode_step call over all layers. The oracle runs, one by one, a
seeded sample of (layer, sequence, kv head) units on the same bytes (the GPU
generates the inputs; the sampled slices are copied to the host).

Per sampled unit: selection scores within SCORE_RTOL, the kept set bit-exact
(near ties excused and counted), codes / fp16 scales / zero-points and the bf16
window bit-exact after prefill and after the last step, and every decode step's
output within the decode tolerance.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import synth
from oracle import OracleCache
from _parity import (DECODE_RTOL, Report, check_export, check_kept, check_scores, decode_error,
                     kvc, np64)


@dataclass
class FullReport(Report):
    units: list = field(default_factory=list)


def _unit_export(ex: dict, b: int, h: int) -> dict:
    """The (b, h) slices of a layer export, as a one-unit export."""
    return {k: v[b:b + 1, h:h + 1] for k, v in ex.items()}


def run_fullsize(spec, steps: int, n_samples: int = 3, seed: int = 0) -> FullReport:
    K = kvc()
    dev = "cuda"
    rep = FullReport()
    L, B, Hk, Hq, D = spec.n_layers, spec.batch, spec.n_kv_heads, spec.n_q_heads, spec.head_dim
    g = spec.gqa
    n, a = spec.prompt_len, spec.obs_window
    ns = n - a
    dims = K.dims_from_spec(spec, max_new_tokens=steps)
    budgets = K.kvc_plan_budgets(dims, spec.schedule, spec.avg_budget, spec.pyramid_depth)
    rng = np.random.default_rng(seed)
    layers = sorted({0, L // 2, L - 1})[:n_samples]
    samples = [(l, int(rng.integers(B)), int(rng.integers(Hk))) for l in layers]
    rep.units = samples
    cache = K.kvc_cache_create(dims, budgets)
    oracles, same = {}, {}
    for l in range(L):
        x = synth.layer_inputs(spec, l, device=dev)
        q_obs = x.get("q_obs")
        cache = K.kvc_prefill_compress(dims, budgets, l, q_obs, x["k"], x["v"], cache=cache)
        scoring = budgets[l] < ns
        mine = [(b, h) for (sl, b, h) in samples if sl == l]
        if not mine:
            continue
        sc = None
        if scoring:
            sc = torch.empty(B, Hk, ns, device=dev)
            K.kvc_scores_layer(cache, sc)
        ex = K.kvc_export_layer(cache, l)
        torch.cuda.synchronize()
        for (b, h) in mine:
            k_np = np64(x["k"][b:b + 1, h:h + 1])
            v_np = np64(x["v"][b:b + 1, h:h + 1])
            q_np = np64(q_obs[b:b + 1, h * g:(h + 1) * g]) if q_obs is not None else None
            oc = OracleCache(1, g, 1, D, spec.bits, spec.group_size, spec.window_len)
            oc.prefill(k_np, v_np, a, budget=budgets[l] if scoring else None, q_obs=q_np,
                       pool_kernel=spec.pool_kernel)
            ok = True
            if scoring:
                check_scores(sc[b, h].double().cpu().numpy(), oc.scores[0][0], rep)
                gk = ex["kept"][b, h].cpu().numpy()
                assert np.all(np.diff(gk) > 0), "kept not ascending"
                ok = check_kept(gk, oc.heads[0][0].kept, oc.pooled[0][0], budgets[l], rep)
            if ok:
                check_export(_unit_export(ex, b, h), oc, [(0, 0)], rep)
            oracles[(l, b, h)] = oc
            same[(l, b, h)] = ok
        del ex
    out = torch.empty(L, B, Hq, D, device=dev)
    for t in range(steps):
        dx = synth.decode_inputs_layers(spec, t, range(L), device=dev)
        K.kvc_decode_step(cache, 0, L, dx["q"], dx["k_new"], dx["v_new"], out)
        for (l, b, h), oc in oracles.items():
            sl = slice(h * g, (h + 1) * g)
            o_ref = oc.step(np64(dx["q"][l, b:b + 1, sl]), np64(dx["k_new"][l, b:b + 1, h:h + 1]),
                            np64(dx["v_new"][l, b:b + 1, h:h + 1]))
            if not same[(l, b, h)]:
                continue
            o_gpu = out[l, b:b + 1, sl].double().cpu().numpy()
            err = decode_error(o_gpu, o_ref)
            rep.decode_err = max(rep.decode_err, err)
            rep.decode_checked += g
            assert err <= DECODE_RTOL, f"unit {(l, b, h)} step {t}: {err:.3g}"
    for (l, b, h), oc in oracles.items():
        info = K.kvc_layer_info_get(cache, l)
        assert info["window_tokens"] == oc.window_len()
        assert info["packed_tokens"] == oc.n_packed()
        if same[(l, b, h)]:
            ex = K.kvc_export_layer(cache, l)
            torch.cuda.synchronize()
            check_export(_unit_export(ex, b, h), oc, [(0, 0)], rep)
            del ex
    K.kvc_check_device(cache)
    cache.close()
    return rep
