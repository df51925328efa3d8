"""The seeded input generators (no method arithmetic): shapes, determinism, and
the full-prompt queries ending in the observation queries."""
import torch

import synth


def test_prompt_queries_shape_seed_and_tail():
    spec = synth.small_spec(2, n_layers=2, batch=2, n_q_heads=8, n_kv_heads=2,
                            prompt_len=300, obs_window=16, avg_budget=64, window_len=64)
    q = synth.prompt_queries(spec, 1)
    assert q.shape == (2, 8, 300, spec.head_dim) and q.dtype == torch.bfloat16
    assert q.is_contiguous()
    assert torch.equal(q, synth.prompt_queries(spec, 1))            # seeded
    assert not torch.equal(q, synth.prompt_queries(spec, 0))        # per layer
    x = synth.layer_inputs(spec, 1)
    assert torch.equal(q[:, :, -16:], x["q_obs"])                   # ends in the window queries
    # the shared per-head direction (queries z + 2 u_h) shows in the mean
    qm = q[:, :, :-16].float().mean(dim=(0, 2))
    assert float(qm.norm(dim=-1).min()) > 1.5


def test_toy_prompt_queries_are_standard_normal():
    spec = synth.workload(1)
    q = synth.prompt_queries(spec, 0).float()
    assert q.shape == (1, 4, 512, 64)
    assert abs(float(q.mean())) < 0.02 and abs(float(q.std()) - 1.0) < 0.02
