"""Selection by MiniKV's full-prompt cumulated attention on the GPU (MiniKV §4.3
"selective flash-attention", Figure 9): scores, kept sets, packed store, window
and decode against the oracle on small cases (ragged row and key blocks, GQA
groups 1-8, pooling on and off, 2- and 4-bit), and sampled columns plus bounds
at the Llama-3-8B prompt length."""
import numpy as np
import pytest
import torch

import synth
from _parity import SCORE_RTOL, kvc, np64, run_small
from oracle import acumul_columns

pytestmark = pytest.mark.gpu

CASES = {
    # GQA 4 (32 positions per row block), n = 1000: ragged row and key blocks
    "gqa4": (synth.small_spec(2, n_layers=2, batch=2, n_q_heads=8, n_kv_heads=2,
                              prompt_len=1000, obs_window=32, avg_budget=96,
                              schedule="uniform", window_len=64), 20),
    # MHA (128 positions per row block), d = 64, no pooling
    "mha_d64_nopool": (synth.small_spec(3, n_layers=1, batch=1, n_q_heads=4, n_kv_heads=4,
                                        head_dim=64, prompt_len=700, obs_window=16,
                                        avg_budget=160, schedule="uniform", pool_kernel=1,
                                        window_len=64), 20),
    # GQA 8 (16 positions per row block), pyramid over 2 layers
    "gqa8": (synth.small_spec(2, n_layers=2, batch=1, n_q_heads=16, n_kv_heads=2,
                              prompt_len=1500, obs_window=16, avg_budget=128,
                              window_len=64), 20),
    # GQA 2, 4-bit
    "gqa2_4bit": (synth.small_spec(2, n_layers=1, batch=1, n_q_heads=4, n_kv_heads=2,
                                   prompt_len=777, obs_window=16, avg_budget=128,
                                   schedule="uniform", bits=4, window_len=96), 20),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_attention_parity(name):
    """The selective flash-attention (MiniKV §4.3, Figure 9): the prefill attention
    output X_O of every query against the oracle, and the selection, store and
    decode it feeds exactly as for kvc_prefill_acumul."""
    spec, steps = CASES[name]
    rep = run_small(spec, steps, selection="attention")
    print(f"{name}: X_O elements={rep.xo_checked} worst |err|/max|v|={rep.xo_err:.2e} "
          f"excused={rep.excused} score_err={rep.score_err:.2e} decode_err={rep.decode_err:.2e}")
    assert rep.xo_checked > 0 and rep.kept_compared > 0 and rep.decode_checked > 0


@pytest.mark.parametrize("name", list(CASES))
def test_acumul_parity(name):
    spec, steps = CASES[name]
    rep = run_small(spec, steps, selection="acumul")
    print(f"{name}: excused={rep.excused} kept_sets={rep.kept_compared} "
          f"codes={rep.codes_compared} decode_err={rep.decode_err:.2e} "
          f"score_err={rep.score_err:.2e}")
    assert rep.kept_compared > 0 and rep.decode_checked > 0


def test_acumul_full_prompt_length_sampled():
    """Llama-3-8B prompt (32,768 tokens, GQA 4, 8 kv heads): every score within
    [0, g (n - j)]; for two units, the first key block's and the last scored
    block's columns against the oracle evaluated column by column."""
    K = kvc()
    spec = synth.workload(2)
    n, a, g = spec.prompt_len, spec.obs_window, spec.gqa
    ns = n - a
    dims = K.dims_from_spec(spec, max_new_tokens=4)
    budgets = K.kvc_plan_budgets(dims, spec.schedule, spec.avg_budget, spec.pyramid_depth)
    cache = K.kvc_cache_create(dims, budgets)
    x = synth.layer_inputs(spec, 0, device="cuda")
    qf = synth.prompt_queries(spec, 0, device="cuda")
    K.kvc_prefill_acumul(cache, 0, qf, x["k"], x["v"])
    sc = torch.empty(spec.batch, spec.n_kv_heads, ns, device="cuda")
    K.kvc_scores_layer(cache, sc)
    K.kvc_check_device(cache)
    s = sc.double().cpu().numpy()
    bound = g * (n - np.arange(ns))
    assert np.all(s >= 0) and np.all(s <= bound * (1 + 1e-5))
    rng = np.random.default_rng(0)
    cols = np.concatenate([np.sort(rng.choice(128, 6, replace=False)),
                           np.sort(rng.choice(np.arange(ns - 96, ns), 6, replace=False))])
    worst = 0.0
    for h in (0, int(rng.integers(1, spec.n_kv_heads))):
        want = acumul_columns(np64(qf[0, h * g:(h + 1) * g]), np64(x["k"][0, h]), cols)
        err = np.abs(s[0, h, cols] - want) / want
        worst = max(worst, float(err.max()))
    print(f"sampled columns {cols.tolist()}: worst relative error {worst:.2e}")
    assert worst <= SCORE_RTOL
    cache.close()


def test_acumul_keep_all_needs_no_queries():
    K = kvc()
    spec = synth.small_spec(2, n_layers=1, batch=1, n_q_heads=8, n_kv_heads=2,
                            prompt_len=300, obs_window=16, avg_budget=64, schedule="none",
                            window_len=64)
    dims = K.dims_from_spec(spec, max_new_tokens=4)
    cache = K.kvc_cache_create(dims, K.kvc_plan_budgets(dims, "none", 0))
    x = synth.layer_inputs(spec, 0, device="cuda")
    K.kvc_prefill_acumul(cache, 0, None, x["k"], x["v"])
    info = K.kvc_layer_info_get(cache, 0)
    assert info["n_kept"] == 300 - 16 and info["packed_tokens"] == 256
    K.kvc_check_device(cache)
    cache.close()


def test_prefill_attention_full_prompt_length_sampled_rows():
    """Llama-3-8B prompt (32,768 tokens, GQA 4): X_O of sampled rows of one unit
    (the first key block, the middle, the observation window) against the oracle's
    definition evaluated for those rows only, and the scores equal to those of
    kvc_prefill_acumul on the same inputs."""
    K = kvc()
    spec = synth.workload(2)
    n, a, g, D = spec.prompt_len, spec.obs_window, spec.gqa, spec.head_dim
    ns = n - a
    dims = K.dims_from_spec(spec, max_new_tokens=4)
    budgets = K.kvc_plan_budgets(dims, spec.schedule, spec.avg_budget, spec.pyramid_depth)
    x = synth.layer_inputs(spec, 0, device="cuda")
    qf = synth.prompt_queries(spec, 0, device="cuda")
    cache = K.kvc_cache_create(dims, budgets)
    xo = torch.empty(spec.batch, spec.n_q_heads, n, D, dtype=torch.bfloat16, device="cuda")
    K.kvc_prefill_attention(cache, 0, qf, x["k"], x["v"], xo)
    sc = torch.empty(spec.batch, spec.n_kv_heads, ns, device="cuda")
    K.kvc_scores_layer(cache, sc)
    kept = K.kvc_export_layer(cache, 0)["kept"]
    K.kvc_check_device(cache)
    cache.close()
    ref_cache = K.kvc_cache_create(dims, budgets)
    K.kvc_prefill_acumul(ref_cache, 0, qf, x["k"], x["v"])
    sc_ref = torch.empty_like(sc)
    K.kvc_scores_layer(ref_cache, sc_ref)
    kept_ref = K.kvc_export_layer(ref_cache, 0)["kept"]
    ref_cache.close()
    rel = ((sc - sc_ref).abs() / sc_ref.abs().clamp_min(1e-30)).max().item()
    assert rel <= 1e-5, rel
    diff = (kept != kept_ref).sum().item()
    print(f"scores vs kvc_prefill_acumul: {rel:.2e}; kept indices differing: {diff}")
    assert diff <= 8            # summation order of the atomics: near-ties only
    rng = np.random.default_rng(1)
    rows = np.concatenate([[0, 1, 127, 128], rng.choice(np.arange(129, ns), 6, replace=False),
                           [ns, n - 1]])
    h = 3
    k64, v64 = np64(x["k"][0, h]), np64(x["v"][0, h])
    worst = 0.0
    for hh in range(g):
        q = np64(qf[0, h * g + hh])
        for i in rows:
            s_ = k64[:i + 1] @ q[i] / np.sqrt(D)
            w = np.exp(s_ - s_.max())
            ref = (w / w.sum()) @ v64[:i + 1]
            got = np64(xo[0, h * g + hh, i])
            vmax = np.abs(v64[:i + 1]).max()
            err = np.abs(got - ref)
            assert np.all(err <= 2.0 ** -8 * (vmax + np.abs(ref))), (hh, i, err.max())
            worst = max(worst, float(err.max() / vmax))
    print(f"sampled rows {rows.tolist()}: worst |err|/max|v| {worst:.2e}")


def test_acumul_scores_are_deterministic():
    """The row blocks' contributions are added as fixed-point integers: three runs
    on the same inputs give bit-identical scores and kept sets (for both the
    selection-only kernel and the one that also forms X_O)."""
    K = kvc()
    spec = CASES["gqa4"][0]
    n, a = spec.prompt_len, spec.obs_window
    dims = K.dims_from_spec(spec, max_new_tokens=4)
    budgets = K.kvc_plan_budgets(dims, spec.schedule, spec.avg_budget, spec.pyramid_depth)
    x = synth.layer_inputs(spec, 0, device="cuda")
    qf = synth.prompt_queries(spec, 0, device="cuda")
    xo = torch.empty(spec.batch, spec.n_q_heads, n, spec.head_dim, dtype=torch.bfloat16,
                     device="cuda")
    cache = K.kvc_cache_create(dims, budgets)
    for call in ("acumul", "attention"):
        runs = []
        for _ in range(3):
            K.kvc_cache_reset(cache)
            if call == "acumul":
                K.kvc_prefill_acumul(cache, 0, qf, x["k"], x["v"])
            else:
                K.kvc_prefill_attention(cache, 0, qf, x["k"], x["v"], xo)
            sc = torch.empty(spec.batch, spec.n_kv_heads, n - a, device="cuda")
            K.kvc_scores_layer(cache, sc)
            runs.append((sc, K.kvc_export_layer(cache, 0)["kept"]))
        torch.cuda.synchronize()
        for sc, kept in runs[1:]:
            assert torch.equal(sc, runs[0][0]), f"{call}: scores differ between runs"
            assert torch.equal(kept, runs[0][1]), f"{call}: kept sets differ between runs"
    K.kvc_check_device(cache)
    cache.close()
