"""The allocation-free selection entry point (kvc_select_noalloc) against the
regular prefill path (kvc_prefill_compress), through the C ABI.

kvc_select_noalloc exists for callers that cannot allocate device memory (they
own all of it through their own arena, or cannot afford a cudaMalloc in the
loop); its intermediates live in a static device array shared by every call.
The test makes two calls in a row on different inputs, so stale contents left
by the first call in that shared array would show up in the second, and checks
the defining property: after a first call on the device, further calls leave
the device's free memory unchanged. It runs last (file name) so that a failure
here leaves every other test already run.
"""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

SCORE_RTOL = 1e-4


SPECS = {
    # GQA 4, head_dim 128
    "gqa4_d128": synth.small_spec(2, n_layers=2, batch=2, n_q_heads=8, n_kv_heads=2,
                                  prompt_len=3000, obs_window=32, avg_budget=256,
                                  schedule="uniform", window_len=64),
    # MHA (g = 1), head_dim 64
    "mha_d64": synth.small_spec(2, n_layers=2, batch=1, n_q_heads=4, n_kv_heads=4, head_dim=64,
                                prompt_len=1500, obs_window=16, avg_budget=128,
                                schedule="uniform", window_len=64),
}


@pytest.mark.parametrize("name", list(SPECS))
def test_select_noalloc_matches_prefill_two_calls(name):
    import kv_cache_compression_snapkv_gb300 as K
    spec = SPECS[name]
    dims = K.dims_from_spec(spec, max_new_tokens=4)
    budgets = K.kvc_plan_budgets(dims, spec.schedule, spec.avg_budget, spec.pyramid_depth)
    B, H, ns = spec.batch, spec.n_kv_heads, spec.prompt_len - spec.obs_window
    cache = None
    for layer in (0, 1):                      # two calls in a row, different inputs
        x = synth.layer_inputs(spec, layer, device="cuda")
        cache = K.kvc_prefill_compress(dims, budgets, layer, x["q_obs"], x["k"], x["v"],
                                       cache=cache)
        ref_scores = torch.empty(B, H, ns, device="cuda")
        K.kvc_scores_layer(cache, ref_scores)
        ref_kept = K.kvc_export_layer(cache, layer)["kept"]

        kept = torch.full((B, H, budgets[layer]), -1, dtype=torch.int32, device="cuda")
        scores = torch.full((B, H, ns), float("nan"), device="cuda")
        K.kvc_select_noalloc(dims, budgets[layer], x["q_obs"], x["k"], kept, scores)
        torch.cuda.synchronize()
        assert torch.equal(kept, ref_kept), f"layer {layer}: kept positions differ"
        torch.testing.assert_close(scores, ref_scores, rtol=SCORE_RTOL, atol=0.0)

        # without the optional scores output (the scores then live in the scratch
        # too); the device's free memory does not move across the call
        kept2 = torch.full_like(kept, -1)
        free0, _ = torch.cuda.mem_get_info()
        K.kvc_select_noalloc(dims, budgets[layer], x["q_obs"], x["k"], kept2)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0, f"free device memory moved by {free0 - free1} bytes"
        assert torch.equal(kept2, ref_kept)
    K.kvc_select_noalloc_check()          # no bounded wait gave up
    cache.close()


def test_select_noalloc_rejects_sizes_beyond_the_scratch():
    import kv_cache_compression_snapkv_gb300 as K
    # 64 sequences x 8 kv heads x 131,072 tokens needs far more than 32 MiB
    dims = K.make_dims(1, 64, 32, 8, 128, 131072, 64, 7, 2, 32, 128, 1)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    kept = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(K.KvcError) as e:
        K.kvc_select_noalloc(dims, 1024, dummy, dummy, kept)
    assert e.value.status == 6          # KVC_E_CAPACITY, nothing enqueued
