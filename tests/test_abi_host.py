"""Host-side checks of the C ABI (no GPU needed): symbols, planner, validation."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "kv_cache_compression_snapkv_gb300", "libkvc.so")


def _header_functions():
    text = open(os.path.join(ROOT, "include", "kvc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def kvc():
    if not os.path.exists(LIB):
        pytest.skip("libkvc.so not built")
    import kv_cache_compression_snapkv_gb300 as k
    return k


def test_library_exports_every_declared_symbol(kvc):
    lib = ctypes.CDLL(LIB)
    names = _header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(kvc.exported_symbols())


def test_named_entry_points_present():
    names = _header_functions()
    for n in ("kvc_plan_budgets", "kvc_prefill_compress", "kvc_append", "kvc_decode_attn",
              "kvc_free"):
        assert n in names


@pytest.mark.parametrize("L,sched,avg,depth,n,alpha", [
    (32, "pyramid", 512, 8, 32768, 32), (32, "pyramid", 1024, 8, 131072, 64),
    (32, "uniform", 128, 0, 8192, 32), (40, "none", 0, 0, 32768, 0),
    (7, "pyramid", 96, 3, 500, 16), (33, "pyramid", 2048, 20, 4096, 8),
    (5, "pyramid", 512, 8, 300, 16), (1, "pyramid", 64, 2, 1000, 8)])
def test_planner_matches_oracle(kvc, L, sched, avg, depth, n, alpha):
    from oracle import plan_budgets
    dims = kvc.make_dims(L, 1, 8, 8, 128, n, alpha, 7, 2, 32, 128, 16)
    got = kvc.kvc_plan_budgets(dims, sched, avg, depth)
    want = plan_budgets(L, sched, avg, depth, 32, max_budget=n - alpha) if sched != "none" \
        else [min(n, n - alpha)] * L
    assert got == want


def test_planner_rejects(kvc):
    dims = kvc.make_dims(4, 1, 8, 8, 128, 1000, 16, 7, 2, 32, 128, 16)
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_plan_budgets(dims, "uniform", 100)
    assert e.value.status == 1
    with pytest.raises(kvc.KvcError):
        kvc.kvc_plan_budgets(dims, "pyramid", 128, 0)


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 96, 2), ("bits", 3, 1), ("group_size", 16, 1), ("n_q_heads", 12, 2),
    ("window_len", 48, 2), ("pool_kernel", 4, 1), ("obs_window", 1000, 2),
    ("obs_window", 200, 2)])
def test_invalid_dims_rejected_before_device_work(kvc, field, value, status):
    base = dict(n_layers=2, batch=1, n_q_heads=8, n_kv_heads=2, head_dim=128, prompt_len=1000,
                obs_window=16, pool_kernel=7, bits=2, group_size=32, window_len=128,
                max_new_tokens=8)
    base[field] = value
    dims = kvc.make_dims(**base)
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_prefill_compress(dims, [64, 64], 0, None, None, None, stream=0)
    assert e.value.status in (status, 1)


def test_null_handles(kvc):
    lib = ctypes.CDLL(LIB)
    lib.kvc_append.restype = ctypes.c_int
    assert lib.kvc_append(None, 0, None, None, None) == 1
    lib.kvc_free.restype = ctypes.c_int
    assert lib.kvc_free(None) == 0
    lib.kvc_status_string.restype = ctypes.c_char_p
    assert lib.kvc_status_string(6) == b"capacity exceeded"


@pytest.mark.parametrize("L,avg,n,alpha,seed,sigma", [
    (32, 512, 32768, 32, 0, 1.0), (32, 1024, 131072, 64, 1, 0.5), (7, 96, 500, 16, 2, 2.0),
    (40, 128, 32768, 32, 3, 1.0), (5, 512, 300, 16, 4, 1.0), (1, 64, 1000, 8, 5, 1.0),
    (32, 512, 32768, 32, 6, 8.0)])
def test_weighted_planner_matches_oracle(kvc, L, avg, n, alpha, seed, sigma):
    """Var-prop / Var-inv budgets: the C planner equals the oracle's on the same
    doubles (exact integers), including weights spanning many decades."""
    from oracle import plan_budgets_weighted, variance_weights
    dims = kvc.make_dims(L, 1, 8, 8, 128, n, alpha, 7, 2, 32, 128, 16)
    var = list(np.random.default_rng(seed).lognormal(0.0, sigma, L))
    for policy in ("var-prop", "var-inv"):
        w = variance_weights(var, policy)
        assert kvc.kvc_plan_budgets_weighted(dims, avg, w) == \
            plan_budgets_weighted(L, avg, w, 32, max_budget=n - alpha)


def test_weighted_planner_rounding_ties(kvc):
    """Weights whose scaled values land on exact halves and equal remainders."""
    from oracle import plan_budgets_weighted
    dims = kvc.make_dims(4, 1, 8, 8, 128, 100000, 32, 7, 2, 32, 128, 16)
    for w in ([1.0, 1.0, 1.0, 1.0], [3.0, 1.0, 1.0, 1.0], [1.0, 2.0 ** -31, 2.0 ** -31, 1.0],
              [1.0, 1.5 * 2.0 ** -30, 2.5 * 2.0 ** -30, 0.75]):
        for avg in (32, 64, 96, 1024):
            assert kvc.kvc_plan_budgets_weighted(dims, avg, w) == \
                plan_budgets_weighted(4, avg, w, 32, max_budget=100000 - 32), (w, avg)


def test_weighted_planner_rejects(kvc):
    dims = kvc.make_dims(3, 1, 8, 8, 128, 1000, 16, 7, 2, 32, 128, 16)
    for w, avg in (([1.0, 0.0, 1.0], 64), ([1.0, float("nan"), 1.0], 64),
                   ([1.0, -1.0, 1.0], 64), ([1.0, 1.0, 1.0], 48)):
        with pytest.raises(kvc.KvcError) as e:
            kvc.kvc_plan_budgets_weighted(dims, avg, w)
        assert e.value.status == 1


def test_new_entry_points_reject_null_handles(kvc):
    lib = ctypes.CDLL(LIB)
    for name, args in (("kvc_prefill_acumul", (None, 0, None, None, None, None)),
                       ("kvc_score_variance", (None, None, None)),
                       ("kvc_plan_budgets_weighted", (None, 64, None, None))):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        assert f(*args) in (1, 2), name       # KVC_E_ARG (or KVC_E_SHAPE for null dims)
