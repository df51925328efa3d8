"""Parity at the workloads' full sizes, in the launch configuration the benchmark
times: every layer compressed with one kvc_prefill_compress call, every decode
step one kvc_decode_step call over all layers.

Two kinds of units are checked against the oracle on the same bytes (the GPU
generates the inputs; the slices are copied to the host):

  * sampled units (at least 8 per workload, spread over the layers, layers 0,
    L/2 and L-1 always among them): selection scores, the kept set (bit-exact,
    near ties excused and counted; an excused unit is then stored by the oracle
    on the GPU's kept set), codes / fp16 scales / zero-points and the bf16 window
    bit-exact after prefill and after the last step, and every decode step's
    output within the decode tolerance;
  * store units (every kv head of every layer where the oracle finishes in
    seconds; a subset of layers and sequences of the quantize-only workload,
    whose 6,400 units hold 32,768 tokens each): the oracle stores the GPU's
    kept set (the selection itself is checked on the sampled units) and replays
    every appended token; codes, scales, zero-points and the window are compared
    bit-exact after prefill and after the last step.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import synth
from oracle import OracleCache
from _parity import (DECODE_RTOL, Report, check_export, check_kept, check_scores, decode_error,
                     kvc, np64, planted_positions)


@dataclass
class FullReport(Report):
    units: list = field(default_factory=list)
    store_units: int = 0


def _unit_export(ex: dict, b: int, h: int) -> dict:
    """The (b, h) slices of a layer export, as a one-unit export."""
    return {k: v[b:b + 1, h:h + 1] for k, v in ex.items()}


def _sampled_units(spec, n_samples, rng):
    L, B, Hk = spec.n_layers, spec.batch, spec.n_kv_heads
    layers = sorted({0, L // 2, L - 1} | {int(x) for x in np.linspace(0, L - 1, n_samples)})
    out = []
    while len(out) < n_samples:
        for l in layers:
            u = (l, int(rng.integers(B)), int(rng.integers(Hk)))
            if u not in out:
                out.append(u)
            if len(out) >= n_samples:
                break
    return out


def _store_units(spec):
    L, B, Hk = spec.n_layers, spec.batch, spec.n_kv_heads
    if spec.prompt_len * B * Hk * L > 64 * 1024 * 1024:   # the quantize-only workload
        return {(l, 0, h) for l in sorted({0, L // 2, L - 1}) for h in range(Hk)}
    if B * Hk * L > 1024:                                 # many short sequences
        return {(l, b, h) for l in range(L) for b in sorted({0, B - 1}) for h in range(Hk)}
    return {(l, b, h) for l in range(L) for b in range(B) for h in range(Hk)}


def run_fullsize(spec, steps: int, n_samples: int = 8, seed: int = 0) -> FullReport:
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
    samples = _sampled_units(spec, n_samples, rng)
    stores = _store_units(spec) - set(samples)
    rep.units = samples
    cache = K.kvc_cache_create(dims, budgets)
    oracles = {}
    for l in range(L):
        x = synth.layer_inputs(spec, l, device=dev)
        q_obs = x.get("q_obs")
        cache = K.kvc_prefill_compress(dims, budgets, l, q_obs, x["k"], x["v"], cache=cache)
        scoring = budgets[l] < ns
        mine = [(b, h) for (sl, b, h) in samples if sl == l]
        store = [(b, h) for (sl, b, h) in stores if sl == l]
        if not mine and not store:
            continue
        sc = None
        if scoring and mine:
            sc = torch.empty(B, Hk, ns, device=dev)
            K.kvc_scores_layer(cache, sc)
        ex = K.kvc_export_layer(cache, l)
        torch.cuda.synchronize()
        for (b, h) in mine + store:
            k_np = np64(x["k"][b:b + 1, h:h + 1])
            v_np = np64(x["v"][b:b + 1, h:h + 1])
            oc = OracleCache(1, g, 1, D, spec.bits, spec.group_size, spec.window_len)
            gk = ex["kept"][b, h].cpu().numpy().astype(np.int64) if scoring else None
            if (b, h) in mine:
                q_np = np64(q_obs[b:b + 1, h * g:(h + 1) * g]) if q_obs is not None else None
                oc.prefill(k_np, v_np, a, budget=budgets[l] if scoring else None, q_obs=q_np,
                           pool_kernel=spec.pool_kernel)
                if scoring:
                    check_scores(sc[b, h].double().cpu().numpy(), oc.scores[0][0], rep,
                                 planted_positions(x, b, h))
                    assert np.all(np.diff(gk) > 0), "kept not ascending"
                    if not check_kept(gk, oc.heads[0][0].kept, oc.pooled[0][0], budgets[l], rep):
                        # an excused near-tie: the oracle stores the GPU's selection
                        rep.rebuilt_units += 1
                        oc = OracleCache(1, g, 1, D, spec.bits, spec.group_size, spec.window_len)
                        oc.prefill(k_np, v_np, a, kept=[[gk]])
            else:
                oc.prefill(k_np, v_np, a, kept=None if gk is None else [[gk]])
                rep.store_units += 1
            check_export(_unit_export(ex, b, h), oc, [(0, 0)], rep)
            oracles[(l, b, h)] = oc
        del ex
    out = torch.empty(L, B, Hq, D, device=dev)
    for t in range(steps):
        dx = synth.decode_inputs_layers(spec, t, range(L), device=dev)
        K.kvc_decode_step(cache, 0, L, dx["q"], dx["k_new"], dx["v_new"], out)
        kn_h, vn_h = dx["k_new"].cpu(), dx["v_new"].cpu()
        o_h = None
        for (l, b, h), oc in oracles.items():
            kn = np64(kn_h[l, b:b + 1, h:h + 1])
            vn = np64(vn_h[l, b:b + 1, h:h + 1])
            if (l, b, h) not in samples:
                oc.append(kn, vn)
                continue
            if o_h is None:
                o_h = out.double().cpu().numpy()
            sl = slice(h * g, (h + 1) * g)
            o_ref = oc.step(np64(dx["q"][l, b:b + 1, sl]), kn, vn)
            err = decode_error(o_h[l, b:b + 1, sl], o_ref)
            rep.decode_err = max(rep.decode_err, err)
            rep.decode_checked += g
            assert err <= DECODE_RTOL, f"unit {(l, b, h)} step {t}: {err:.3g}"
    layers_done = {}
    for (l, b, h), oc in oracles.items():
        info = K.kvc_layer_info_get(cache, l)
        assert info["window_tokens"] == oc.window_len()
        assert info["packed_tokens"] == oc.n_packed()
        if l not in layers_done:
            layers_done.clear()
            layers_done[l] = K.kvc_export_layer(cache, l)
            torch.cuda.synchronize()
        check_export(_unit_export(layers_done[l], b, h), oc, [(0, 0)], rep)
    layers_done.clear()
    K.kvc_check_device(cache)
    cache.close()
    return rep
