"""Host-side validation of the C ABI, checked without a GPU: every entry point
rejects a null cache handle; cache creation validates per-layer precisions,
budgets, ring lengths and the size limits before touching the device; the
allocation-free selection validates its shape and scratch capacity before any
CUDA call. On a machine without a GPU a cache whose dimensions pass validation
fails at the first device call (KVC_E_CUDA), which shows where validation ends."""
import ctypes

import pytest

K = pytest.importorskip("kv_cache_compression_snapkv_gb300")

E_ARG, E_SHAPE, E_CUDA, E_CAPACITY = 1, 2, 4, 6


def _has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


# calls below pass made-up device addresses to checks that must return before any
# launch; on a machine with a GPU a wrong expectation would launch with them
host_only = pytest.mark.skipif(_has_gpu(), reason="host-only checks with made-up pointers")


def _dims(**kw):
    base = dict(n_layers=4, batch=1, n_q_heads=8, n_kv_heads=2, head_dim=128, prompt_len=4096,
                obs_window=32, pool_kernel=7, bits=2, group_size=32, window_len=128,
                max_new_tokens=64)
    base.update(kw)
    return K.make_dims(**base)


def _create(dims, budgets, layer_bits=None):
    h = ctypes.c_void_p()
    b = (ctypes.c_int32 * len(budgets))(*budgets)
    if layer_bits is None:
        st = K._lib.kvc_cache_create(ctypes.byref(dims), b, ctypes.byref(h))
    else:
        lb = (ctypes.c_int32 * len(layer_bits))(*layer_bits)
        st = K._lib.kvc_cache_create_layers(ctypes.byref(dims), b, lb, ctypes.byref(h))
    assert st != 0 or h.value, "a created cache has a handle"
    if st == 0:
        K._lib.kvc_free(h)
    return st


def test_every_entry_point_rejects_a_null_cache():
    P = ctypes.c_void_p(256)   # never dereferenced: the null cache is rejected first
    lib = K._lib
    calls = {
        "kvc_prefill_selected": (None, 0, P, 32, P, P, None),
        "kvc_prefill_sinks": (None, 0, 4, P, P, None),
        "kvc_prefill_acumul": (None, 0, P, P, P, None),
        "kvc_prefill_attention": (None, 0, P, P, P, P, None),
        "kvc_append": (None, 0, P, P, None),
        "kvc_append_layers": (None, 0, 1, P, P, None),
        "kvc_decode_attn": (None, 0, 1, P, P, None),
        "kvc_decode_step": (None, 0, 1, P, P, P, P, None),
        "kvc_layer_info_get": (None, 0, ctypes.byref(K.KvcLayerInfo())),
        "kvc_export_layer": (None, 0, ctypes.byref(K.KvcExport()), None),
        "kvc_scores_layer": (None, P, P, None),
        "kvc_score_variance": (None, P, None),
        "kvc_cache_reset": (None,),
        "kvc_check_device": (None, None),
        "kvc_set_wait_limit": (None, 0),
    }
    for name, args in calls.items():
        assert getattr(lib, name)(*args) == E_ARG, name
    assert lib.kvc_free(None) == 0
    dims = _dims()
    b = (ctypes.c_int32 * 4)(64, 64, 64, 64)
    assert lib.kvc_cache_create(ctypes.byref(dims), b, None) == E_ARG
    assert lib.kvc_cache_create_layers(ctypes.byref(dims), b, None, None) == E_ARG
    h = ctypes.c_void_p()
    assert lib.kvc_cache_create_layers(ctypes.byref(dims), b, None, ctypes.byref(h)) == E_ARG
    assert lib.kvc_cache_create(ctypes.byref(dims), None, ctypes.byref(h)) == E_ARG


@pytest.mark.parametrize("layer_bits", [[2, 4, 3, 2], [2, 0, 2, 2], [8, 2, 2, 2], [2, 2, 2, -16]])
def test_create_layers_rejects_unknown_precisions(layer_bits):
    assert _create(_dims(), [64] * 4, layer_bits) == E_ARG


def test_create_rejects_negative_budgets():
    assert _create(_dims(), [64, -32, 64, 64]) == E_ARG


def test_sixteen_bit_ring_limits():
    # a 16-bit layer inside a 2-bit cache gets a ring for its kept, observation and
    # appended tokens: at most 65,536 slots
    ok = _dims(max_new_tokens=65536 - 32 - 1024)
    big = _dims(max_new_tokens=65536 - 32 - 1024 + 1)
    assert _create(big, [1024] * 4, [2, 2, 16, 2]) == E_SHAPE
    # the largest max_new_tokens: a long ring, rejected; past the limit (where the
    # ring arithmetic would once have wrapped to a short ring), rejected up front
    for m in (1 << 24, (1 << 24) + 1, (1 << 31) - 1):
        assert _create(_dims(max_new_tokens=m), [1024] * 4, [2, 2, 16, 2]) == E_SHAPE, m
        assert _create(_dims(bits=16, window_len=65536, max_new_tokens=m), [1024] * 4) \
            == E_SHAPE, m
    if not _has_gpu():
        assert _create(ok, [1024] * 4, [2, 2, 16, 2]) == E_CUDA
    # a cache stored at 16 bits throughout: window_len must hold them itself
    all16 = _dims(bits=16, window_len=1024 + 32 + 64)
    assert _create(all16, [1024] * 4) in ((E_CUDA,) if not _has_gpu() else (0,))
    short = _dims(bits=16, window_len=1024 + 32 + 32)
    assert _create(short, [1024] * 4) == E_SHAPE


def test_initial_window_must_fit_its_ring():
    # 2-bit: the kept tokens past the last whole group plus the observation tokens
    # must leave room in the ring (budget 64 + 16 keeps 16 past the last group)
    dims = _dims(n_q_heads=2, obs_window=112, window_len=128)
    assert _create(dims, [80] * 4) == E_SHAPE
    if not _has_gpu():
        assert _create(dims, [64] * 4) == E_CUDA


def test_scoring_rows_limited():
    # a scoring layer needs g * obs_window <= 256 rows (here 4 * 96 = 384)
    dims = _dims(obs_window=96, window_len=256)
    assert _create(dims, [64] * 4) == E_SHAPE
    # keep-all layers score nothing, so the limit does not apply
    if not _has_gpu():
        assert _create(dims, [4096 - 96] * 4) == E_CUDA


@pytest.mark.parametrize("field,value", [
    ("prompt_len", (1 << 30) + 1), ("max_new_tokens", (1 << 24) + 1), ("batch", (1 << 21) + 1),
    ("prompt_len", 0), ("n_layers", 257)])
def test_size_limits(field, value):
    dims = _dims(**{field: value})
    with pytest.raises(K.KvcError) as e:
        K.kvc_plan_budgets(dims, "uniform", 64)
    assert e.value.status == E_SHAPE


def test_size_limits_inclusive():
    for field, value in (("prompt_len", 1 << 30), ("max_new_tokens", 1 << 24),
                         ("batch", 1 << 21)):
        dims = _dims(**{field: value})
        assert len(K.kvc_plan_budgets(dims, "uniform", 64)) == 4, field


def test_allocator_hooks_come_in_pairs():
    dims = _dims()
    dims.alloc = K._alloc_fn(lambda n, s, c: None)
    assert _create(dims, [64] * 4) == E_ARG


@host_only
@pytest.mark.parametrize("kw,budget,status", [
    (dict(n_q_heads=6, n_kv_heads=2), 64, E_SHAPE),          # g = 3
    (dict(head_dim=96), 64, E_SHAPE),
    (dict(prompt_len=1, obs_window=0), 64, E_SHAPE),
    (dict(obs_window=0), 64, E_SHAPE),
    (dict(obs_window=4096), 64, E_SHAPE),
    (dict(obs_window=96), 64, E_SHAPE),                       # g * alpha = 384 > 256
    (dict(pool_kernel=4), 64, E_ARG),
    (dict(), -1, E_ARG),
    (dict(batch=4097, n_kv_heads=2), 64, E_CAPACITY),         # more than 8,192 units
    (dict(batch=16, prompt_len=131072, obs_window=64), 64, E_CAPACITY),   # > 32 MiB
])
def test_select_noalloc_validation(kw, budget, status):
    P = ctypes.c_void_p(256)   # made-up addresses: every case returns before a launch
    dims = _dims(**kw)
    assert K._lib.kvc_select_noalloc(ctypes.byref(dims), budget, P, P, P, None, None) == status


@host_only
def test_select_noalloc_null_arguments():
    P = ctypes.c_void_p(256)
    dims = _dims()
    f = K._lib.kvc_select_noalloc
    assert f(None, 64, P, P, P, None, None) == E_ARG
    assert f(ctypes.byref(dims), 64, None, P, P, None, None) == E_ARG
    assert f(ctypes.byref(dims), 64, P, None, P, None, None) == E_ARG
    assert f(ctypes.byref(dims), 64, P, P, None, None, None) == E_ARG


@host_only
def test_select_noalloc_without_a_device():
    # valid dimensions within the scratch: the first CUDA call fails on this machine
    P = ctypes.c_void_p(256)
    dims = _dims()
    assert K._lib.kvc_select_noalloc(ctypes.byref(dims), 64, P, P, P, None, None) == E_CUDA


@host_only
def test_prefill_compress_checks_its_arguments_before_creating_a_cache():
    """With *cache NULL, a call whose own arguments are invalid returns KVC_E_ARG
    and creates nothing (on a machine without a GPU, creation would fail with
    KVC_E_CUDA, so KVC_E_ARG shows the check came first)."""
    P = ctypes.c_void_p(256)   # made-up addresses: every case returns before a launch
    dims = _dims()
    f = K._lib.kvc_prefill_compress
    scoring = (ctypes.c_int32 * 4)(64, 64, 64, 64)
    keep_all = (ctypes.c_int32 * 4)(*([4096 - 32] * 4))
    for budgets, layer, q, k, v in ((scoring, 0, P, None, P), (scoring, 0, P, P, None),
                                    (scoring, 4, P, P, P), (scoring, -1, P, P, P),
                                    (scoring, 0, None, P, P), (None, 0, P, P, P)):
        h = ctypes.c_void_p()
        assert f(ctypes.byref(dims), budgets, layer, q, k, v, ctypes.byref(h), None) == E_ARG
        assert h.value is None, "nothing created"
    # a keep-all layer needs no observation queries: creation is reached
    h = ctypes.c_void_p()
    assert f(ctypes.byref(dims), keep_all, 0, None, P, P, ctypes.byref(h), None) == E_CUDA
    assert h.value is None
