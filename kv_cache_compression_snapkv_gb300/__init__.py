"""Compressed-KV-cache attention for GB300: Python binding of libkvc.so.

Thin ctypes marshalling over the C ABI in include/kvc.h -- the functions keep
the C names; every step of the path runs in the library's CUDA kernels. PyTorch
only supplies device memory and streams. Importing fails loudly if the library
has not been built (`python -m kv_cache_compression_snapkv_gb300._build`).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
# KVC_LIB selects another build of the library (e.g. libkvc_checked.so, with
# device-side index checks); by default the one built next to this file.
LIB_PATH = os.environ.get("KVC_LIB") or os.path.join(_HERE, "libkvc.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -m kv_cache_compression_snapkv_gb300._build)")

_lib = ctypes.CDLL(LIB_PATH)

# ----------------------------------------------------------------- C types
KVC_OK = 0
STATUS_NAMES = {0: "KVC_OK", 1: "KVC_E_ARG", 2: "KVC_E_SHAPE", 3: "KVC_E_OOM", 4: "KVC_E_CUDA",
                5: "KVC_E_STATE", 6: "KVC_E_CAPACITY", 7: "KVC_E_TIMEOUT",
                8: "KVC_E_DEVICE_CHECK"}
SCHED = {"none": 0, "uniform": 1, "pyramid": 2}

_alloc_fn = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p)
_free_fn = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p)


class KvcDims(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("prompt_len", ctypes.c_int32),
                ("obs_window", ctypes.c_int32), ("pool_kernel", ctypes.c_int32),
                ("bits", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("window_len", ctypes.c_int32), ("max_new_tokens", ctypes.c_int32),
                ("alloc", _alloc_fn), ("free", _free_fn), ("alloc_ctx", ctypes.c_void_p)]


class KvcLayerInfo(ctypes.Structure):
    _fields_ = [("prefilled", ctypes.c_int32), ("budget", ctypes.c_int32),
                ("n_kept", ctypes.c_int32), ("packed_tokens", ctypes.c_int32),
                ("capacity_tokens", ctypes.c_int32), ("window_tokens", ctypes.c_int32),
                ("appended", ctypes.c_int32), ("packed_bytes", ctypes.c_int64),
                ("bits", ctypes.c_int32), ("window_capacity", ctypes.c_int32)]


class KvcExport(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in
                ("kept", "k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero",
                 "win_k", "win_v")]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_S = ctypes.c_int
_SIGS = {
    "kvc_plan_budgets": [ctypes.POINTER(KvcDims), _S, _I, _I, _P],
    "kvc_plan_budgets_weighted": [ctypes.POINTER(KvcDims), _I, _P, _P],
    "kvc_prefill_compress": [ctypes.POINTER(KvcDims), _P, _I, _P, _P, _P,
                             ctypes.POINTER(ctypes.c_void_p), _P],
    "kvc_prefill_selected": [_P, _I, _P, _I, _P, _P, _P],
    "kvc_prefill_sinks": [_P, _I, _I, _P, _P, _P],
    "kvc_prefill_acumul": [_P, _I, _P, _P, _P, _P],
    "kvc_prefill_attention": [_P, _I, _P, _P, _P, _P, _P],
    "kvc_cache_create": [ctypes.POINTER(KvcDims), _P, ctypes.POINTER(ctypes.c_void_p)],
    "kvc_cache_create_layers": [ctypes.POINTER(KvcDims), _P, _P, ctypes.POINTER(ctypes.c_void_p)],
    "kvc_append": [_P, _I, _P, _P, _P],
    "kvc_append_layers": [_P, _I, _I, _P, _P, _P],
    "kvc_decode_attn": [_P, _I, _I, _P, _P, _P],
    "kvc_decode_step": [_P, _I, _I, _P, _P, _P, _P, _P],
    "kvc_free": [_P],
    "kvc_layer_info_get": [_P, _I, ctypes.POINTER(KvcLayerInfo)],
    "kvc_export_layer": [_P, _I, ctypes.POINTER(KvcExport), _P],
    "kvc_scores_layer": [_P, _P, _P, _P],
    "kvc_score_variance": [_P, _P, _P],
    "kvc_cache_reset": [_P],
    "kvc_select_noalloc": [ctypes.POINTER(KvcDims), _I, _P, _P, _P, _P, _P],
    "kvc_select_noalloc_check": [_P],
    "kvc_check_device": [_P, _P],
    "kvc_set_wait_limit": [_P, ctypes.c_int64],
}
for _name, _args in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
_lib.kvc_build_checked.argtypes = []
_lib.kvc_build_checked.restype = ctypes.c_int32
_lib.kvc_launch_count.argtypes = []
_lib.kvc_launch_count.restype = ctypes.c_uint64
_lib.kvc_status_string.argtypes = [ctypes.c_int]
_lib.kvc_status_string.restype = ctypes.c_char_p


class KvcError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call}: {STATUS_NAMES.get(status, status)} "
                         f"({_lib.kvc_status_string(status).decode()})")


def _check(status: int, call: str):
    if status != KVC_OK:
        raise KvcError(status, call)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def make_dims(n_layers, batch, n_q_heads, n_kv_heads, head_dim, prompt_len, obs_window,
              pool_kernel, bits, group_size, window_len, max_new_tokens) -> KvcDims:
    return KvcDims(n_layers, batch, n_q_heads, n_kv_heads, head_dim, prompt_len, obs_window,
                   pool_kernel, bits, group_size, window_len, max_new_tokens)


def dims_from_spec(spec, max_new_tokens: Optional[int] = None) -> KvcDims:
    """kvc_dims of a synthetic workload description (any object with the fields)."""
    return make_dims(spec.n_layers, spec.batch, spec.n_q_heads, spec.n_kv_heads, spec.head_dim,
                     spec.prompt_len, spec.obs_window, spec.pool_kernel, spec.bits,
                     spec.group_size, spec.window_len,
                     spec.steps if max_new_tokens is None else max_new_tokens)


# ------------------------------------------------------------------ the ABI
def kvc_plan_budgets(dims: KvcDims, schedule: str, avg_budget: int,
                     pyramid_depth: int = 0) -> list:
    out = (ctypes.c_int32 * dims.n_layers)()
    _check(_lib.kvc_plan_budgets(ctypes.byref(dims), SCHED[schedule], avg_budget, pyramid_depth,
                                 out), "kvc_plan_budgets")
    return list(out)


def kvc_plan_budgets_weighted(dims: KvcDims, avg_budget: int, weights: Sequence[float]) -> list:
    """Budgets in proportion to per-layer weights (Var-prop: the layers' variance
    scores; Var-inv: their inverses)."""
    if len(weights) != dims.n_layers:
        raise ValueError("need one weight per layer")
    w = (ctypes.c_double * dims.n_layers)(*[float(x) for x in weights])
    out = (ctypes.c_int32 * dims.n_layers)()
    _check(_lib.kvc_plan_budgets_weighted(ctypes.byref(dims), avg_budget, w, out),
           "kvc_plan_budgets_weighted")
    return list(out)


class Cache:
    """Owner of a kvc_cache* (freed by close() or garbage collection)."""

    def __init__(self, handle: int, dims: KvcDims, budgets: Sequence[int]):
        self.handle = handle
        self.dims = dims
        self.budgets = list(budgets)

    def close(self):
        if self.handle:
            _lib.kvc_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _budget_array(budgets):
    return (ctypes.c_int32 * len(budgets))(*budgets)


def kvc_cache_create(dims: KvcDims, budgets: Sequence[int]) -> Cache:
    h = ctypes.c_void_p()
    _check(_lib.kvc_cache_create(ctypes.byref(dims), _budget_array(budgets), ctypes.byref(h)),
           "kvc_cache_create")
    return Cache(h.value, dims, budgets)


def kvc_cache_create_layers(dims: KvcDims, budgets: Sequence[int],
                            layer_bits: Sequence[int]) -> Cache:
    """A cache whose layers have their own precision (2, 4 or 16 bits each)."""
    if len(layer_bits) != dims.n_layers:
        raise ValueError("need one precision per layer")
    h = ctypes.c_void_p()
    _check(_lib.kvc_cache_create_layers(ctypes.byref(dims), _budget_array(budgets),
                                        _budget_array(list(layer_bits)), ctypes.byref(h)),
           "kvc_cache_create_layers")
    return Cache(h.value, dims, budgets)


def kvc_prefill_compress(dims: KvcDims, budgets: Sequence[int], layer: int, q_obs, k, v,
                         cache: Optional[Cache] = None, stream=None) -> Cache:
    h = ctypes.c_void_p(cache.handle if cache is not None else None)
    st = _lib.kvc_prefill_compress(ctypes.byref(dims), _budget_array(budgets), layer,
                                   _ptr(q_obs), _ptr(k), _ptr(v), ctypes.byref(h),
                                   _stream(stream))
    if st != KVC_OK and cache is None and h.value:
        _lib.kvc_free(h.value)    # created by this call, which then failed
    _check(st, "kvc_prefill_compress")
    return cache if cache is not None else Cache(h.value, dims, budgets)


def kvc_prefill_selected(cache: Cache, layer: int, kept, n_kept: int, k, v, stream=None):
    _check(_lib.kvc_prefill_selected(cache.handle, layer, _ptr(kept), n_kept, _ptr(k), _ptr(v),
                                     _stream(stream)), "kvc_prefill_selected")


def kvc_prefill_sinks(cache: Cache, layer: int, n_sinks: int, k, v, stream=None):
    """Attention-sink + recent-token selection of `layer` (no scoring), then packing."""
    _check(_lib.kvc_prefill_sinks(cache.handle, layer, n_sinks, _ptr(k), _ptr(v),
                                  _stream(stream)), "kvc_prefill_sinks")


def kvc_prefill_acumul(cache: Cache, layer: int, q_full, k, v, stream=None):
    """Selection of `layer` by MiniKV's full-prompt cumulated attention (every
    prompt query, un-normalised column sums), then packing."""
    _check(_lib.kvc_prefill_acumul(cache.handle, layer, _ptr(q_full), _ptr(k), _ptr(v),
                                   _stream(stream)), "kvc_prefill_acumul")


def kvc_prefill_attention(cache: Cache, layer: int, q_full, k, v, x_out, stream=None):
    """MiniKV's selective flash-attention of `layer`: the causal attention output of
    every prompt query into x_out (bf16 [B][Hq][n][d]) and, from the same tiles, the
    selection by the cumulated attention, then packing."""
    _check(_lib.kvc_prefill_attention(cache.handle, layer, _ptr(q_full), _ptr(k), _ptr(v),
                                      _ptr(x_out), _stream(stream)), "kvc_prefill_attention")


def kvc_append(cache: Cache, layer: int, k_new, v_new, stream=None):
    _check(_lib.kvc_append(cache.handle, layer, _ptr(k_new), _ptr(v_new), _stream(stream)),
           "kvc_append")


def kvc_append_layers(cache: Cache, layer_begin: int, layer_count: int, k_new, v_new,
                      stream=None):
    _check(_lib.kvc_append_layers(cache.handle, layer_begin, layer_count, _ptr(k_new),
                                  _ptr(v_new), _stream(stream)), "kvc_append_layers")


def kvc_decode_attn(cache: Cache, layer_begin: int, layer_count: int, q, out, stream=None):
    _check(_lib.kvc_decode_attn(cache.handle, layer_begin, layer_count, _ptr(q), _ptr(out),
                                _stream(stream)), "kvc_decode_attn")


def kvc_decode_step(cache: Cache, layer_begin: int, layer_count: int, q, k_new, v_new, out,
                    stream=None):
    _check(_lib.kvc_decode_step(cache.handle, layer_begin, layer_count, _ptr(q), _ptr(k_new),
                                _ptr(v_new), _ptr(out), _stream(stream)), "kvc_decode_step")


def kvc_free(cache: Cache):
    cache.close()


def kvc_layer_info_get(cache: Cache, layer: int) -> dict:
    info = KvcLayerInfo()
    _check(_lib.kvc_layer_info_get(cache.handle, layer, ctypes.byref(info)), "kvc_layer_info_get")
    return {name: getattr(info, name) for name, _ in KvcLayerInfo._fields_}


def kvc_export_layer(cache: Cache, layer: int, stream=None) -> dict:
    """Unpack one layer into fresh device tensors (see include/kvc.h)."""
    import torch
    info = kvc_layer_info_get(cache, layer)
    d = cache.dims
    B, H, D = d.batch, d.n_kv_heads, d.head_dim
    T, W, K = info["packed_tokens"], info["window_tokens"], info["n_kept"]
    dev = torch.device("cuda", torch.cuda.current_device())
    out = {
        "kept": torch.empty(B, H, K, dtype=torch.int32, device=dev),
        "k_codes": torch.empty(B, H, T, D, dtype=torch.uint8, device=dev),
        "k_scale": torch.empty(B, H, T // 32, D, dtype=torch.float16, device=dev),
        "k_zero": torch.empty(B, H, T // 32, D, dtype=torch.float16, device=dev),
        "v_codes": torch.empty(B, H, T, D, dtype=torch.uint8, device=dev),
        "v_scale": torch.empty(B, H, T, D // 32, dtype=torch.float16, device=dev),
        "v_zero": torch.empty(B, H, T, D // 32, dtype=torch.float16, device=dev),
        "win_k": torch.empty(B, H, W, D, dtype=torch.bfloat16, device=dev),
        "win_v": torch.empty(B, H, W, D, dtype=torch.bfloat16, device=dev),
    }
    ex = KvcExport(*[(_ptr(out[n]) if out[n].numel() else None)
                     for n, _ in KvcExport._fields_])
    _check(_lib.kvc_export_layer(cache.handle, layer, ctypes.byref(ex), _stream(stream)),
           "kvc_export_layer")
    return out


def kvc_scores_layer(cache: Cache, scores=None, pooled=None, stream=None):
    _check(_lib.kvc_scores_layer(cache.handle, _ptr(scores), _ptr(pooled), _stream(stream)),
           "kvc_scores_layer")


def kvc_score_variance(cache: Cache, var_out, stream=None):
    """Per-(sequence, kv head) variance of the last scored layer's selection
    scores into var_out (device fp32 [B][H])."""
    _check(_lib.kvc_score_variance(cache.handle, _ptr(var_out), _stream(stream)),
           "kvc_score_variance")


def kvc_cache_reset(cache: Cache):
    _check(_lib.kvc_cache_reset(cache.handle), "kvc_cache_reset")


def kvc_select_noalloc(dims: KvcDims, budget: int, q_obs, k, kept, scores=None, stream=None):
    """Selection of one layer into `kept` (and `scores`) without any device
    allocation; intermediates use the library's static 32 MiB device scratch."""
    _check(_lib.kvc_select_noalloc(ctypes.byref(dims), budget, _ptr(q_obs), _ptr(k), _ptr(kept),
                                   _ptr(scores), _stream(stream)), "kvc_select_noalloc")


def kvc_select_noalloc_check(stream=None):
    """Synchronize and raise KvcError(KVC_E_TIMEOUT) if a bounded wait of a
    kvc_select_noalloc call on this device gave up since the last check."""
    _check(_lib.kvc_select_noalloc_check(_stream(stream)), "kvc_select_noalloc_check")


def kvc_check_device(cache: Cache, stream=None):
    """Synchronize and raise KvcError(KVC_E_DEVICE_CHECK) if a check of the checked
    build found an index out of range, KvcError(KVC_E_TIMEOUT) if a bounded device wait
    gave up."""
    _check(_lib.kvc_check_device(cache.handle, _stream(stream)), "kvc_check_device")


def kvc_set_wait_limit(cache: Cache, polls: int):
    """Bound the cache's decode staging waits to `polls` polls (negative: default)."""
    _check(_lib.kvc_set_wait_limit(cache.handle, polls), "kvc_set_wait_limit")


def kvc_launch_count() -> int:
    return int(_lib.kvc_launch_count())


def kvc_build_checked() -> bool:
    """True if the loaded library was built with device-side index checks."""
    return bool(_lib.kvc_build_checked())


def exported_symbols() -> list:
    """Names of the C entry points this binding resolved."""
    return sorted(list(_SIGS) + ["kvc_status_string", "kvc_launch_count", "kvc_build_checked"])


__all__ = ["KvcDims", "KvcError", "Cache", "make_dims", "dims_from_spec", "kvc_plan_budgets",
           "kvc_cache_create", "kvc_cache_create_layers", "kvc_prefill_compress", "kvc_prefill_selected", "kvc_prefill_sinks",
           "kvc_append",
           "kvc_append_layers", "kvc_decode_attn", "kvc_decode_step", "kvc_free",
           "kvc_layer_info_get", "kvc_export_layer", "kvc_scores_layer", "kvc_cache_reset",
           "kvc_plan_budgets_weighted", "kvc_score_variance", "kvc_prefill_acumul",
           "kvc_prefill_attention",
           "kvc_launch_count", "kvc_check_device", "kvc_build_checked", "kvc_select_noalloc",
           "kvc_select_noalloc_check", "kvc_set_wait_limit", "LIB_PATH",
           "exported_symbols"]
