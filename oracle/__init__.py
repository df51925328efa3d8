"""CPU oracle for compressed-KV-cache attention -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct numpy restatement of what the hot path computes,
written from the pages' statement of the method:

  * budgets.py     per-layer token budgets (uniform / PyramidKV-style linear)
  * snapkv.py      observation-window scores, 1-D max-pooling, per-head top-k
  * acumul.py      full-prompt cumulated attention (MiniKV's A_cumul: column sums
                   of un-normalised FlashAttention tiles) and its selection
  * sinks.py       attention-sink + recent-token selection (StreamingLLM-style)
  * variance.py    variance score of a layer's selection scores and the
                   variance-driven budgets (Var-prop / Var-inv)
  * quant.py       KIVI-style asymmetric group quantization (keys per channel,
                   values per token), b = 2 or 4 bits, fp16 scale and zero-point
  * cache.py       the compressed cache: prefill selection + quantization, the
                   bf16 recent window with group-by-group flushing, and decode
                   attention over packed + window tokens
  * arithmetic.py  cache-size arithmetic printed on the pages

Floating point is fp64 except where the method fixes the precision: the group
quantizer runs in fp32 with IEEE round-to-nearest division and round-half-to-even
codes and stores fp16 scale/zero-point.

This package shares no code with the CUDA library (`kv_cache_compression_snapkv_gb300`)
and neither imports the other. Only `tests/`, `__graft_entry__.smoke()` and the
CPU-baseline leg of `bench.py` may import it; the product path never routes here.
"""
from .budgets import plan_budgets
from .snapkv import window_scores, max_pool, select_topk, snapkv_select
from .sinks import sinks_window_select
from .acumul import acumul_scores, acumul_select, acumul_columns, prefill_attention
from .variance import (score_variance, layer_variance, variance_weights,
                       plan_budgets_weighted)
from .quant import (quantize_group, quantize_keys, quantize_values, dequantize_keys,
                    dequantize_values)
from .cache import OracleCache
from .arithmetic import (blog_budget_row, minikv_sizes)

__all__ = [
    "plan_budgets", "window_scores", "max_pool", "select_topk", "snapkv_select",
    "sinks_window_select", "acumul_scores", "acumul_select", "acumul_columns", "score_variance", "layer_variance", "variance_weights",
    "plan_budgets_weighted",
    "quantize_group", "quantize_keys", "quantize_values", "dequantize_keys",
    "dequantize_values", "OracleCache", "blog_budget_row",
    "minikv_sizes",
]
