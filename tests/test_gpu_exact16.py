"""16-bit storage (bits = 16: no quantization, every kept token stays exact in the
bf16 window) on the GPU.

With every prompt token kept, the cache must reduce to plain dense attention: the
decode output of each step equals softmax(q . K^T / sqrt(d)) V over all prompt
tokens and all tokens appended so far, computed here directly in fp64 from the
same bf16 inputs (no oracle code involved). With a SnapKV selection (the oracle's
kept positions given to the GPU), the decode output matches the oracle's 16-bit
cache.
"""
import math

import numpy as np
import pytest
import torch

import synth
from _parity import DECODE_RTOL, decode_error, kvc, np64
from oracle import OracleCache

pytestmark = pytest.mark.gpu


def _ceil32(x):
    return (x + 31) // 32 * 32


def test_full_budget_is_dense_attention():
    K = kvc()
    steps = 20
    spec = synth.small_spec(2, n_layers=2, batch=1, n_q_heads=8, n_kv_heads=2,
                            prompt_len=1000, obs_window=32, schedule="none", bits=16,
                            window_len=_ceil32(1000 + steps))
    L, B, Hq, Hk, D, n = (spec.n_layers, spec.batch, spec.n_q_heads, spec.n_kv_heads,
                          spec.head_dim, spec.prompt_len)
    g = Hq // Hk
    dims = K.dims_from_spec(spec, max_new_tokens=steps)
    budgets = K.kvc_plan_budgets(dims, "none", 0)
    cache = None
    keys, vals = [], []
    for l in range(L):
        x = synth.layer_inputs(spec, l, device="cpu", with_q=False)
        cache = K.kvc_prefill_compress(dims, budgets, l, None, x["k"].cuda(), x["v"].cuda(),
                                       cache=cache)
        keys.append(np64(x["k"]))
        vals.append(np64(x["v"]))
    for l in range(L):
        info = K.kvc_layer_info_get(cache, l)
        assert info["packed_tokens"] == 0 and info["window_tokens"] == n
    worst = 0.0
    for t in range(steps):
        dx = synth.decode_inputs_layers(spec, t, range(L), device="cpu")
        out = torch.empty(L, B, Hq, D, device="cuda")
        K.kvc_decode_step(cache, 0, L, dx["q"].cuda(), dx["k_new"].cuda(), dx["v_new"].cuda(), out)
        torch.cuda.synchronize()
        for l in range(L):
            keys[l] = np.concatenate([keys[l], np64(dx["k_new"][l])[:, :, None]], axis=2)
            vals[l] = np.concatenate([vals[l], np64(dx["v_new"][l])[:, :, None]], axis=2)
            q = np64(dx["q"][l])                                   # [B][Hq][D]
            ref = np.empty((B, Hq, D))
            for b in range(B):
                for h in range(Hq):
                    kk, vv = keys[l][b, h // g], vals[l][b, h // g]
                    s = kk @ q[b, h] / math.sqrt(D)
                    w = np.exp(s - s.max())
                    ref[b, h] = (w / w.sum()) @ vv
            err = decode_error(out[l].double().cpu().numpy(), ref)
            worst = max(worst, err)
            assert err <= DECODE_RTOL, f"layer {l} step {t}: {err:.3g}"
    print(f"dense equivalence: worst relative error {worst:.2e} over {steps} steps")
    K.kvc_check_device(cache)
    cache.close()


def test_selected_tokens_stay_exact():
    K = kvc()
    steps = 12
    spec = synth.small_spec(2, n_layers=1, batch=1, n_q_heads=4, n_kv_heads=1,
                            prompt_len=700, obs_window=16, avg_budget=160, bits=16,
                            window_len=_ceil32(160 + 16 + steps))
    B, Hq, Hk, D, n, a = (spec.batch, spec.n_q_heads, spec.n_kv_heads, spec.head_dim,
                          spec.prompt_len, spec.obs_window)
    dims = K.dims_from_spec(spec, max_new_tokens=steps)
    budgets = K.kvc_plan_budgets(dims, spec.schedule, spec.avg_budget, spec.pyramid_depth)
    x = synth.layer_inputs(spec, 0, device="cpu")
    oc = OracleCache(B, Hq, Hk, D, 16, spec.group_size, spec.window_len)
    oc.prefill(np64(x["k"]), np64(x["v"]), a, budget=budgets[0], q_obs=np64(x["q_obs"]),
               pool_kernel=spec.pool_kernel)
    cache = K.kvc_cache_create(dims, budgets)
    kept = torch.tensor(np.stack([[oc.heads[b][h].kept for h in range(Hk)] for b in range(B)]),
                        dtype=torch.int32, device="cuda")
    K.kvc_prefill_selected(cache, 0, kept, kept.shape[-1], x["k"].cuda(), x["v"].cuda())
    worst = 0.0
    for t in range(steps):
        dx = synth.decode_inputs_layers(spec, t, [0], device="cpu")
        out = torch.empty(1, B, Hq, D, device="cuda")
        K.kvc_decode_step(cache, 0, 1, dx["q"].cuda(), dx["k_new"].cuda(), dx["v_new"].cuda(), out)
        torch.cuda.synchronize()
        ref = oc.step(np64(dx["q"][0]), np64(dx["k_new"][0]), np64(dx["v_new"][0]))
        err = decode_error(out[0].double().cpu().numpy(), ref)
        worst = max(worst, err)
        assert err <= DECODE_RTOL, f"step {t}: {err:.3g}"
    ex = K.kvc_export_layer(cache, 0)
    torch.cuda.synchronize()
    st = oc.heads[0][0]
    # the window holds the kept tokens, the observation tokens and the appended ones, exact
    exact_rows = np.concatenate([st.k_hat, st.win_k])
    np.testing.assert_array_equal(np64(ex["win_k"][0, 0]), exact_rows)
    print(f"16-bit selection: worst relative error {worst:.2e}")
    cache.close()
