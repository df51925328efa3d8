"""Error paths of the C ABI on the GPU: a failing allocator hook, calls out of
order, capacity, argument checks, and the bounded-wait timeout path of the decode
kernel (driven by a zero wait limit: every staging wait gives up at once, so no
GPU ever hangs or faults), after which the cache is reset and must give exactly
the outputs of a fresh cache."""

import pytest
import torch

import synth
from _parity import kvc

pytestmark = pytest.mark.gpu

SPEC = synth.small_spec(2, n_layers=2, batch=1, n_q_heads=8, n_kv_heads=2, prompt_len=1000,
                        obs_window=32, avg_budget=96, window_len=64)

E_ARG, E_OOM, E_STATE, E_CAPACITY, E_TIMEOUT = 1, 3, 5, 6, 7


def _status(fn, *args):
    K = kvc()
    try:
        fn(*args)
    except K.KvcError as e:
        return e.status
    return 0


def _prefilled(steps, spec=SPEC):
    K = kvc()
    dims = K.dims_from_spec(spec, max_new_tokens=steps)
    budgets = K.kvc_plan_budgets(dims, spec.schedule, spec.avg_budget, spec.pyramid_depth)
    cache = None
    prompt = []
    for l in range(spec.n_layers):
        x = synth.layer_inputs(spec, l, device="cuda")
        prompt.append(x)
        cache = K.kvc_prefill_compress(dims, budgets, l, x["q_obs"], x["k"], x["v"], cache=cache)
    return K, dims, budgets, cache, prompt


def _step_inputs(t, spec=SPEC):
    dx = synth.decode_inputs_layers(spec, t, range(spec.n_layers), device="cuda")
    return dx["q"], dx["k_new"], dx["v_new"]


def test_failing_allocator_reports_oom_and_frees_the_rest():
    K = kvc()
    live, counts = {}, {"alloc": 0, "free": 0}
    limit = 3          # the fourth allocation of the cache fails

    def alloc(nbytes, stream, ctx):
        if counts["alloc"] >= limit:
            return None
        t = torch.empty(int(nbytes), dtype=torch.uint8, device="cuda")
        live[t.data_ptr()] = t
        counts["alloc"] += 1
        return t.data_ptr()

    def free(ptr, stream, ctx):
        counts["free"] += 1
        live.pop(ptr)

    cb_alloc, cb_free = K._alloc_fn(alloc), K._free_fn(free)
    dims = K.dims_from_spec(SPEC, max_new_tokens=4)
    dims.alloc, dims.free = cb_alloc, cb_free
    budgets = K.kvc_plan_budgets(dims, SPEC.schedule, SPEC.avg_budget, SPEC.pyramid_depth)
    assert _status(K.kvc_cache_create, dims, budgets) == E_OOM
    assert counts["alloc"] == limit and counts["free"] == limit and not live


def test_calls_out_of_order_and_past_capacity():
    K = kvc()
    dims = K.dims_from_spec(SPEC, max_new_tokens=3)
    budgets = K.kvc_plan_budgets(dims, SPEC.schedule, SPEC.avg_budget, SPEC.pyramid_depth)
    cache = K.kvc_cache_create(dims, budgets)
    q, kn, vn = _step_inputs(0)
    out = torch.empty(SPEC.n_layers, SPEC.batch, SPEC.n_q_heads, SPEC.head_dim, device="cuda")
    # decode / append before prefill
    assert _status(K.kvc_decode_step, cache, 0, SPEC.n_layers, q, kn, vn, out) == E_STATE
    assert _status(K.kvc_decode_attn, cache, 0, 1, q[0], out[0]) == E_STATE
    assert _status(K.kvc_append, cache, 0, kn[0], vn[0]) == E_STATE
    cache.close()
    K, dims, budgets, cache, _ = _prefilled(3)
    # a layer compressed twice
    x = synth.layer_inputs(SPEC, 0, device="cuda")
    assert _status(K.kvc_prefill_compress, dims, budgets, 0, x["q_obs"], x["k"], x["v"],
                   cache) == E_STATE
    for t in range(3):
        q, kn, vn = _step_inputs(t)
        K.kvc_decode_step(cache, 0, SPEC.n_layers, q, kn, vn, out)
    q, kn, vn = _step_inputs(3)
    assert _status(K.kvc_decode_step, cache, 0, SPEC.n_layers, q, kn, vn, out) == E_CAPACITY
    assert _status(K.kvc_append, cache, 1, kn[1], vn[1]) == E_CAPACITY
    # misaligned query / output (bulk copies and vector stores need 16 bytes)
    qb = torch.empty(q.numel() + 8, dtype=q.dtype, device="cuda")
    assert _status(K.kvc_decode_attn, cache, 0, 1, qb[1:1 + q[0].numel()], out[0]) == E_ARG
    ob = torch.empty(out.numel() + 4, device="cuda")
    assert _status(K.kvc_decode_attn, cache, 0, 1, q[0], ob[1:1 + out[0].numel()]) == E_ARG
    # a range of layers outside the model
    assert _status(K.kvc_decode_attn, cache, 1, 2, q, out) == E_ARG
    K.kvc_check_device(cache)
    cache.close()


def test_timeout_is_reported_and_the_cache_recovers():
    steps = 6
    K, dims, budgets, cache, prompt = _prefilled(steps)
    L, B, Hq, D = SPEC.n_layers, SPEC.batch, SPEC.n_q_heads, SPEC.head_dim
    out = torch.empty(L, B, Hq, D, device="cuda")
    K.kvc_set_wait_limit(cache, 0)          # every staging wait gives up at once
    q, kn, vn = _step_inputs(0)
    K.kvc_decode_step(cache, 0, L, q, kn, vn, out)   # enqueued; the kernel winds down
    torch.cuda.synchronize()
    # reported by the next call on the cache (host-visible error word) or else by
    # kvc_check_device; either way exactly once
    first = _status(K.kvc_decode_attn, cache, 0, L, q, out)
    if first == 0:
        assert _status(K.kvc_check_device, cache) == E_TIMEOUT
    else:
        assert first == E_TIMEOUT
    assert _status(K.kvc_check_device, cache) == 0
    # recovery: default bound, reset, prefill again; the outputs must equal a fresh
    # cache's bit for bit (the arrival counters of split units returned to zero)
    K.kvc_set_wait_limit(cache, -1)
    K.kvc_cache_reset(cache)
    for l in range(L):
        x = prompt[l]
        K.kvc_prefill_compress(dims, budgets, l, x["q_obs"], x["k"], x["v"], cache=cache)
    fresh = K.kvc_cache_create(dims, budgets)
    for l in range(L):
        x = prompt[l]
        K.kvc_prefill_compress(dims, budgets, l, x["q_obs"], x["k"], x["v"], cache=fresh)
    out2 = torch.empty_like(out)
    for t in range(steps):
        q, kn, vn = _step_inputs(t)
        K.kvc_decode_step(cache, 0, L, q, kn, vn, out)
        K.kvc_decode_step(fresh, 0, L, q, kn, vn, out2)
        torch.cuda.synchronize()
        assert torch.equal(out, out2), f"step {t}: recovered cache differs from a fresh one"
    K.kvc_check_device(cache)
    K.kvc_check_device(fresh)
    cache.close()
    fresh.close()
