"""The checked build (KVC_CHECKED=1): kept positions given to kvc_prefill_selected
are range-checked on the device. A position outside [0, prompt_len - obs_window)
is skipped (position 0 is read in its place) and the next call on the cache
returns KVC_E_DEVICE_CHECK; a valid selection reports nothing. The out-of-range
position used here, prompt_len - obs_window, still lies inside the unit's own key
rows (an observation token), so even an unchecked read of it stays in bounds.

The checked library is built on first use (separate objects, libkvc_checked.so)
and driven in a child process that loads it through KVC_LIB."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "kv_cache_compression_snapkv_gb300")

CHILD = r"""
import sys
import torch
import synth
import kv_cache_compression_snapkv_gb300 as K

assert K._lib.kvc_build_checked() == 1, "not the checked build"
E_DEVICE_CHECK = 8
spec = synth.small_spec(2, n_layers=2, batch=1, n_q_heads=8, n_kv_heads=2, prompt_len=640,
                        obs_window=32, avg_budget=128, window_len=64)
dims = K.dims_from_spec(spec, max_new_tokens=4)
budgets = K.kvc_plan_budgets(dims, "uniform", 128, 0)
ns = spec.prompt_len - spec.obs_window
units = spec.batch * spec.n_kv_heads


def status(fn, *a):
    try:
        fn(*a)
    except K.KvcError as e:
        return e.status
    return 0


for bad in (False, True):
    cache = K.kvc_cache_create(dims, budgets)
    x = synth.layer_inputs(spec, 0, device="cuda")
    kept = torch.arange(0, 4 * 128, 4, dtype=torch.int32, device="cuda")   # < ns
    kept = kept.repeat(units, 1).contiguous()
    if bad:
        kept[0, -1] = ns            # outside the scored range
    K.kvc_prefill_selected(cache, 0, kept, 128, x["k"], x["v"])
    torch.cuda.synchronize()
    y = synth.layer_inputs(spec, 1, device="cuda")
    st = status(K.kvc_prefill_selected, cache, 1, kept[:, :96].contiguous(), 96, y["k"], y["v"])
    if bad:
        # reported by the next call on the cache (host-visible error word) or else by
        # kvc_check_device; either way exactly once
        if st == 0:
            assert status(K.kvc_check_device, cache) == E_DEVICE_CHECK
        else:
            assert st == E_DEVICE_CHECK, st
        assert status(K.kvc_check_device, cache) == 0
    else:
        assert st == 0, st
        assert status(K.kvc_check_device, cache) == 0
    cache.close()
print("checked build ok")
"""


def _checked_library() -> str:
    lib = os.path.join(PKG, "libkvc_checked.so")
    srcs = [os.path.join(PKG, "csrc", f) for f in os.listdir(os.path.join(PKG, "csrc"))]
    srcs.append(os.path.join(ROOT, "include", "kvc.h"))
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(s) for s in srcs):
        sys.path.insert(0, ROOT)
        import importlib.util
        spec = importlib.util.spec_from_file_location("_kvc_build", os.path.join(PKG, "_build.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build(checked=True)
    return lib


def test_normal_build_reports_unchecked():
    sys.path.insert(0, ROOT)
    import kv_cache_compression_snapkv_gb300 as K
    if os.environ.get("KVC_LIB"):
        pytest.skip("KVC_LIB selects another build")
    assert K._lib.kvc_build_checked() == 0


def test_checked_build_reports_out_of_range_kept():
    lib = _checked_library()
    env = dict(os.environ, KVC_LIB=lib, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "checked build ok" in r.stdout
