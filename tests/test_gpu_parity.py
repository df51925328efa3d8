"""CUDA path vs oracle on workloads the oracle finishes in seconds (several key
tiles, ragged tails, every GQA group size, 2- and 4-bit, flushes during decode)."""
import pytest

import synth
from _parity import run_small

pytestmark = pytest.mark.gpu

CASES = {
    # the toy workload at full size: MHA, d=64, window == group (flush at step 16)
    "toy": (synth.workload(1), 20, "score"),
    # GQA g=4, d=128, pyramid over 3 layers (top layer budget 0), ragged n
    "gqa4_pyramid": (synth.small_spec(2, n_layers=3, batch=2, n_q_heads=8, n_kv_heads=2,
                                      prompt_len=1000, obs_window=32, avg_budget=96,
                                      window_len=64), 40, "score"),
    # quantize-only, MHA, 4-bit, prompt not a multiple of the group
    "quant_only_4bit": (synth.small_spec(3, n_layers=2, batch=2, n_q_heads=4, n_kv_heads=4,
                                         prompt_len=300, window_len=64), 60, "score"),
    # g=8 with d=64, uniform budget
    "gqa8_d64": (synth.small_spec(4, n_layers=1, batch=1, n_q_heads=16, n_kv_heads=2,
                                  head_dim=64, prompt_len=700, obs_window=16,
                                  avg_budget=160, window_len=64), 70, "score"),
    # g=2, 4-bit with eviction
    "gqa2_4bit": (synth.small_spec(2, n_layers=2, batch=1, n_q_heads=4, n_kv_heads=2,
                                   prompt_len=777, obs_window=16, avg_budget=128,
                                   schedule="uniform", bits=4, window_len=96), 50, "score"),
    # long-context flavour: M = 256 scoring rows, needles, window 128
    "long_needles": (synth.small_spec(5, n_layers=2, batch=1, n_q_heads=8, n_kv_heads=2,
                                      prompt_len=4096, obs_window=64, avg_budget=256,
                                      window_len=128), 130, "score"),
    # a large budget (4,096 of a 32,768-key prompt kept per head), 4-bit
    "large_budget": (synth.small_spec(2, n_layers=1, batch=1, n_q_heads=2, n_kv_heads=1,
                                      head_dim=64, prompt_len=32800, obs_window=32,
                                      avg_budget=4096, schedule="uniform", bits=4,
                                      window_len=64), 12, "score"),
    # scoring rows not a multiple of 32: M = 2 x 20 = 40 (one partial 32-row chunk of
    # the column sums) and M = 8 x 25 = 200 (two row halves, the second partial)
    "obs20_m40": (synth.small_spec(2, n_layers=2, batch=2, n_q_heads=4, n_kv_heads=2,
                                   prompt_len=900, obs_window=20, avg_budget=128,
                                   window_len=64), 30, "score"),
    "obs25_m200": (synth.small_spec(2, n_layers=1, batch=1, n_q_heads=16, n_kv_heads=2,
                                    prompt_len=1100, obs_window=25, avg_budget=160,
                                    window_len=64), 30, "score"),
    # attention sinks + recent tokens (no scoring), pyramid budgets over 3 layers
    "sinks_window": (synth.small_spec(2, n_layers=3, batch=2, n_q_heads=8, n_kv_heads=2,
                                      prompt_len=1000, obs_window=32, avg_budget=96,
                                      window_len=64), 40, ("sinks", 4)),
    # the GPU given the oracle's selection (storage + decode parity alone)
    "oracle_selection": (synth.small_spec(2, n_layers=2, batch=2, n_q_heads=8, n_kv_heads=2,
                                          prompt_len=1500, obs_window=32, avg_budget=160,
                                          window_len=64), 35, "oracle"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_parity(name):
    spec, steps, selection = CASES[name]
    rep = run_small(spec, steps, selection=selection)
    print(f"{name}: excused={rep.excused} kept_sets={rep.kept_compared} "
          f"codes={rep.codes_compared} decode_err={rep.decode_err:.2e} "
          f"score_err={rep.score_err:.2e}")
    assert rep.decode_checked > 0


def test_per_layer_calls_match():
    """Single-layer append/decode calls give the same results as one multi-layer launch."""
    spec = synth.small_spec(2, n_layers=2, batch=1, n_q_heads=4, n_kv_heads=1,
                            prompt_len=600, obs_window=16, avg_budget=64, window_len=32)
    rep = run_small(spec, 12, selection="score", multi_layer_decode=False)
    assert rep.decode_err <= 2e-3


def test_mixed_precision_layers():
    """One cache whose layers differ in precision (MiniKV Figure 1: 16-bit top
    layers, 2-bit lower ones; here also a 4-bit layer), every decode step one
    launch over all four layers, each layer against the oracle at its own
    precision, across window flushes."""
    spec = synth.small_spec(2, n_layers=4, batch=2, n_q_heads=8, n_kv_heads=2,
                            prompt_len=1000, obs_window=32, avg_budget=96, window_len=64)
    rep = run_small(spec, 45, selection="score", layer_bits=[2, 2, 4, 16])
    print(f"mixed: excused={rep.excused} codes={rep.codes_compared} "
          f"decode_err={rep.decode_err:.2e}")
    assert rep.decode_checked > 0


def test_selected_after_reset_on_a_keep_all_layer():
    """A keep-all layer (budget >= prompt_len - obs_window) has no stored selection
    from creation; kvc_prefill_selected gives it one. After kvc_cache_reset a second
    call with more kept positions must still fit, and its store is compared with
    the oracle's on the same selection (kept set, codes, scales, zero-points and
    window, bit for bit)."""
    import numpy as np
    import torch
    from _parity import Report, check_export, kvc, np64
    from oracle import OracleCache

    K = kvc()
    B, Hq, Hk, D, n, a = 1, 4, 2, 128, 512, 16
    dims = K.make_dims(1, B, Hq, Hk, D, n, a, 7, 2, 32, 64, 4)
    budgets = K.kvc_plan_budgets(dims, "none", 0)
    assert budgets[0] >= n - a
    gen = torch.Generator().manual_seed(91)
    k = torch.randn(B, Hk, n, D, generator=gen).to(torch.bfloat16)
    v = torch.randn(B, Hk, n, D, generator=gen).to(torch.bfloat16)
    rng = np.random.default_rng(91)
    cache = K.kvc_cache_create(dims, budgets)
    try:
        for nk in (64, 200):
            sel = [[np.sort(rng.choice(n - a, nk, replace=False)) for _ in range(Hk)]
                   for _ in range(B)]
            kept = torch.tensor(np.array(sel), dtype=torch.int32, device="cuda")
            K.kvc_cache_reset(cache)
            K.kvc_prefill_selected(cache, 0, kept, nk, k.cuda(), v.cuda())
            ex = K.kvc_export_layer(cache, 0)
            torch.cuda.synchronize()
            oc = OracleCache(B, Hq, Hk, D, 2, 32, 64)
            oc.prefill(np64(k), np64(v), a, kept=sel)
            for b in range(B):
                for h in range(Hk):
                    np.testing.assert_array_equal(ex["kept"][b, h].cpu().numpy(), sel[b][h])
            rep = Report()
            check_export(ex, oc, [(b, h) for b in range(B) for h in range(Hk)], rep)
            assert rep.codes_compared == B * Hk * (nk // 32 * 32)
    finally:
        cache.close()
