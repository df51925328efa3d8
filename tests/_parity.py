"""Shared parity machinery: run a workload through the CUDA path (C ABI) and the
oracle on the same seeded inputs and compare.

Acceptance rules (compressed-KV parity):
  * packed codes, fp16 scales and zero-points: bit-exact;
  * kept index sets: bit-exact, except an index in the symmetric difference is
    excused when its oracle pooled score is within 1e-5 relative of the oracle's
    k-th largest pooled score (fp32 GPU scores vs fp64 oracle scores); a unit
    with an excused difference is then stored by the oracle on the GPU's own
    kept set, so that its codes, window and decode are still compared;
  * selection scores: relative error <= 1e-4, each score against itself with a
    floor of 1e-3 of the largest score of the unit's unplanted keys (planted
    sinks and needles take most of a row's weight and would otherwise hide the
    error on the ordinary keys being ranked);
  * bf16 window: bit-exact;
  * decode output (fp32): max over (sequence, query head, step) of
    ||o - o*||_inf / ||o*||_inf <= 2e-3.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import synth
from oracle import OracleCache, prefill_attention, sinks_window_select

DECODE_RTOL = 2e-3
TIE_RTOL = 1e-5
SCORE_RTOL = 1e-4


def kvc():
    import kv_cache_compression_snapkv_gb300 as k
    return k


@dataclass
class Report:
    excused: int = 0
    kept_compared: int = 0
    codes_compared: int = 0
    decode_err: float = 0.0
    decode_checked: int = 0
    score_err: float = 0.0
    rebuilt_units: int = 0
    xo_err: float = 0.0
    xo_checked: int = 0
    notes: list = field(default_factory=list)


def np64(t):
    return t.detach().float().cpu().double().numpy()


def check_kept(gpu_kept, ora_kept, ora_pooled, k, rep: Report):
    g, o = set(map(int, gpu_kept)), set(map(int, ora_kept))
    diff = g ^ o
    rep.kept_compared += 1
    if not diff:
        return True
    tau = np.sort(ora_pooled)[::-1][k - 1]
    for i in diff:
        assert abs(ora_pooled[i] - tau) <= TIE_RTOL * abs(tau), \
            f"kept sets differ at {i}: pooled {ora_pooled[i]!r} vs k-th {tau!r}"
    rep.excused += len(diff)
    return False


def planted_positions(x: dict, b: int, h: int) -> list:
    """Sink and needle positions of unit (b, h) of synth.layer_inputs' output."""
    pos = list(x.get("sinks") or [])
    if x.get("needles") is not None:
        pos += [int(i) for i in x["needles"][b, h].tolist()]
    return pos


def check_scores(gpu_s, ora_s, rep: Report, planted=()):
    ordinary = np.ones(len(ora_s), dtype=bool)
    ordinary[[p for p in planted if p < len(ora_s)]] = False
    scale = np.abs(ora_s[ordinary]).max() if ordinary.any() else np.abs(ora_s).max()
    err = np.abs(gpu_s - ora_s) / np.maximum(np.abs(ora_s), 1e-3 * scale)
    rep.score_err = max(rep.score_err, float(err.max()))
    assert err.max() <= SCORE_RTOL, f"score error {err.max():.3g}"


def check_export(ex: dict, oc: OracleCache, heads, rep: Report):
    """Bit-exact comparison of one layer's packed store and window. A 16-bit layer
    keeps every token in the GPU's window: the oracle's exact store (its packed
    part, then its window) is compared with it."""
    for (b, h) in heads:
        st = oc.heads[b][h]
        if oc.bits == 16:
            assert ex["k_codes"].shape[2] == 0
            np.testing.assert_array_equal(np64(ex["win_k"][b, h]), np.vstack([st.k_hat, st.win_k]))
            np.testing.assert_array_equal(np64(ex["win_v"][b, h]), np.vstack([st.v_hat, st.win_v]))
            rep.codes_compared += len(st.k_hat) + len(st.win_k)
            continue
        T = st.n_packed
        assert ex["k_codes"].shape[2] == T, (ex["k_codes"].shape, T)
        np.testing.assert_array_equal(ex["k_codes"][b, h].cpu().numpy(), st.kcodes)
        np.testing.assert_array_equal(ex["v_codes"][b, h].cpu().numpy(), st.vcodes)
        for name, ref in (("k_scale", st.kS), ("k_zero", st.kZ), ("v_scale", st.vS),
                          ("v_zero", st.vZ)):
            got = ex[name][b, h].cpu().numpy().view(np.uint16)
            np.testing.assert_array_equal(got, ref.view(np.uint16), err_msg=name)
        np.testing.assert_array_equal(np64(ex["win_k"][b, h]), st.win_k)
        np.testing.assert_array_equal(np64(ex["win_v"][b, h]), st.win_v)
        rep.codes_compared += T


def check_prefill_attention(x_gpu, q_group, k, v, rep: Report):
    """The GPU's X_O of one kv head ([g][n][d], bf16) against the oracle's. The GPU
    rounds the attention weights to bf16 (relative 2^-9) before the product with
    V, and the output to bf16 (relative 2^-9): element by element
    |x - x*| <= 2^-9 (max |v| over the row's keys) + 2^-9 |x*|; tested with 2^-8."""
    ref = prefill_attention(q_group, k, v)
    vmax = np.maximum.accumulate(np.abs(v).max(axis=1))       # max |v| over keys <= i
    bound = 2.0 ** -8 * (vmax[None, :, None] + np.abs(ref))
    err = np.abs(x_gpu - ref)
    rep.xo_err = max(rep.xo_err, float((err / np.maximum(vmax[None, :, None], 1e-30)).max()))
    rep.xo_checked += ref.size
    assert np.all(err <= bound), f"X_O off by {float((err - bound).max()):.3g} over the bound"


def decode_error(o_gpu, o_ora):
    """max over (b, head) of ||o - o*||_inf / ||o*||_inf."""
    diff = np.abs(o_gpu - o_ora).max(axis=-1)
    ref = np.abs(o_ora).max(axis=-1)
    return float((diff / ref).max())


def run_small(spec, steps, selection="score", layers=None, multi_layer_decode=True,
              dev="cuda", budgets=None, layer_bits=None):
    """Full comparison on a workload the oracle finishes in seconds.

    selection: "score" (GPU scores and selects; the oracle does the same),
               "oracle" (the GPU is given the oracle's kept positions) or
               ("sinks", s) (both keep s attention sinks + the most recent tokens) or
               "acumul" (both score by the full-prompt cumulated attention) or
               "attention" (as "acumul", through the selective flash-attention that
               also returns the prefill attention output, checked against the oracle).
    budgets: per-layer budgets to use instead of the spec's schedule.
    layer_bits: per-layer storage precision (2, 4 or 16) of one mixed cache.
    """
    K = kvc()
    rep = Report()
    layers = list(range(spec.n_layers)) if layers is None else layers
    dims = K.dims_from_spec(spec, max_new_tokens=steps)
    if budgets is None:
        budgets = K.kvc_plan_budgets(dims, spec.schedule, spec.avg_budget, spec.pyramid_depth)
    n, a = spec.prompt_len, spec.obs_window
    B, Hk, Hq, D = spec.batch, spec.n_kv_heads, spec.n_q_heads, spec.head_dim
    cache = None if layer_bits is None else K.kvc_cache_create_layers(dims, budgets, layer_bits)
    oracles = {}
    same = {}
    for layer in layers:
        x = synth.layer_inputs(spec, layer, device="cpu")
        k_np, v_np = np64(x["k"]), np64(x["v"])
        q_np = np64(x["q_obs"]) if "q_obs" in x else None
        bud = budgets[layer]
        if layer_bits is None:
            oc = OracleCache(B, Hq, Hk, D, spec.bits, spec.group_size, spec.window_len)
        else:
            ring = K.kvc_layer_info_get(cache, layer)["window_capacity"]
            oc = OracleCache(B, Hq, Hk, D, layer_bits[layer], spec.group_size, ring)
        scoring = bud < n - a
        sinks = selection[1] if isinstance(selection, tuple) else None
        if sinks is not None:
            sel = sinks_window_select(n - a, bud, sinks)
            oc.prefill(k_np, v_np, a, kept=[[sel] * Hk for _ in range(B)])
        else:
            qf = (synth.prompt_queries(spec, layer, device="cpu")
                  if selection in ("acumul", "attention") else None)
            oc.prefill(k_np, v_np, a, budget=bud if scoring else None, q_obs=q_np,
                       pool_kernel=spec.pool_kernel, q_full=None if qf is None else np64(qf))
        kd, vd = x["k"].to(dev), x["v"].to(dev)
        qd = x["q_obs"].to(dev) if "q_obs" in x else None
        if sinks is not None:
            if cache is None:
                cache = K.kvc_cache_create(dims, budgets)
            K.kvc_prefill_sinks(cache, layer, sinks, kd, vd)
            ex = K.kvc_export_layer(cache, layer)
            torch.cuda.synchronize()
            if scoring:
                for b in range(B):
                    for h in range(Hk):
                        np.testing.assert_array_equal(ex["kept"][b, h].cpu().numpy(),
                                                      oc.heads[b][h].kept)
                        rep.kept_compared += 1
            ok_heads = [(b, h) for b in range(B) for h in range(Hk)]
        elif selection == "oracle" or not scoring:
            if cache is None:
                cache = K.kvc_cache_create(dims, budgets)
            nk = len(oc.heads[0][0].kept)
            kept = torch.tensor(np.stack([[oc.heads[b][h].kept for h in range(Hk)]
                                          for b in range(B)]), dtype=torch.int32, device=dev)
            K.kvc_prefill_selected(cache, layer, kept, nk, kd, vd)
            ok_heads = [(b, h) for b in range(B) for h in range(Hk)]
        else:
            if selection == "acumul":
                if cache is None:
                    cache = K.kvc_cache_create(dims, budgets)
                K.kvc_prefill_acumul(cache, layer, qf.to(dev), kd, vd)
            elif selection == "attention":
                if cache is None:
                    cache = K.kvc_cache_create(dims, budgets)
                xo = torch.empty(B, Hq, n, D, dtype=torch.bfloat16, device=dev)
                K.kvc_prefill_attention(cache, layer, qf.to(dev), kd, vd, xo)
                torch.cuda.synchronize()
                g = Hq // Hk
                qf64 = np64(qf)
                for b in range(B):
                    for h in range(Hk):
                        check_prefill_attention(np64(xo[b, h * g:(h + 1) * g]),
                                                qf64[b, h * g:(h + 1) * g], k_np[b, h],
                                                v_np[b, h], rep)
            else:
                cache = K.kvc_prefill_compress(dims, budgets, layer, qd, kd, vd, cache=cache)
            sc = torch.empty(B, Hk, n - a, device=dev)
            pl = torch.empty(B, Hk, n - a, device=dev)
            K.kvc_scores_layer(cache, sc, pl)
            info = K.kvc_layer_info_get(cache, layer)
            ex = K.kvc_export_layer(cache, layer)
            torch.cuda.synchronize()
            ok_heads = []
            for b in range(B):
                for h in range(Hk):
                    check_scores(sc[b, h].double().cpu().numpy(), oc.scores[b][h], rep,
                                 planted_positions(x, b, h))
                    np.testing.assert_array_equal(
                        pl[b, h].double().cpu().numpy(),
                        _pool_of(sc[b, h].double().cpu().numpy(), spec.pool_kernel))
                    gk = ex["kept"][b, h].cpu().numpy()
                    assert np.all(np.diff(gk) > 0), "kept not ascending"
                    if check_kept(gk, oc.heads[b][h].kept, oc.pooled[b][h], bud, rep):
                        ok_heads.append((b, h))
            assert info["n_kept"] == bud
            if len(ok_heads) < B * Hk:
                # an excused near-tie: store the GPU's selection in the oracle too and
                # compare everything downstream of it
                gk_all = [[ex["kept"][b, h].cpu().numpy().astype(np.int64) for h in range(Hk)]
                          for b in range(B)]
                rep.rebuilt_units += B * Hk - len(ok_heads)
                oc = OracleCache(B, Hq, Hk, D, oc.bits, spec.group_size, oc.R)
                oc.prefill(k_np, v_np, a, kept=gk_all)
                ok_heads = [(b, h) for b in range(B) for h in range(Hk)]
        ex = K.kvc_export_layer(cache, layer)
        torch.cuda.synchronize()
        check_export(ex, oc, ok_heads, rep)
        oracles[layer] = oc
        same[layer] = ok_heads
    # decode
    for t in range(steps):
        dx = synth.decode_inputs_layers(spec, t, layers, device="cpu")
        qd, knd, vnd = dx["q"].to(dev), dx["k_new"].to(dev), dx["v_new"].to(dev)
        out = torch.empty(len(layers), B, Hq, D, device=dev)
        contiguous = layers == list(range(layers[0], layers[0] + len(layers)))
        if multi_layer_decode and contiguous:
            K.kvc_decode_step(cache, layers[0], len(layers), qd, knd, vnd, out)
        else:
            for i, layer in enumerate(layers):
                K.kvc_append(cache, layer, knd[i], vnd[i])
                K.kvc_decode_attn(cache, layer, 1, qd[i], out[i])
        torch.cuda.synchronize()
        for i, layer in enumerate(layers):
            o_ref = oracles[layer].step(np64(dx["q"][i]), np64(dx["k_new"][i]),
                                        np64(dx["v_new"][i]))
            o_gpu = out[i].double().cpu().numpy()
            g = spec.gqa
            for (b, h) in same[layer]:
                sl = slice(h * g, (h + 1) * g)
                err = decode_error(o_gpu[b, sl], o_ref[b, sl])
                rep.decode_err = max(rep.decode_err, err)
                rep.decode_checked += g
                assert err <= DECODE_RTOL, f"layer {layer} step {t} (b={b},h={h}): {err:.3g}"
    # final state matches after the flushes
    for layer in layers:
        info = K.kvc_layer_info_get(cache, layer)
        if oracles[layer].bits == 16:
            assert info["packed_tokens"] == 0
            assert info["window_tokens"] == oracles[layer].n_packed() + oracles[layer].window_len()
        else:
            assert info["window_tokens"] == oracles[layer].window_len()
            assert info["packed_tokens"] == oracles[layer].n_packed()
        ex = K.kvc_export_layer(cache, layer)
        torch.cuda.synchronize()
        check_export(ex, oracles[layer], same[layer], rep)
    K.kvc_check_device(cache)          # no bounded device wait gave up
    cache.close()
    return rep


def _pool_of(s, w):
    """Max-pool used only to check the GPU's pooled copy against its own scores."""
    r = (w - 1) // 2
    out = np.empty_like(s)
    for i in range(len(s)):
        out[i] = s[max(0, i - r):i + r + 1].max()
    return out
