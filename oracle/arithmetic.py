"""Cache-size arithmetic printed on the pages -- oracle (test infrastructure only).

Follows:
  * KV Cache Compression: Eviction and Quantization (blog), "The budget": bytes
    per token of context = 2 (K and V) * layers * kv heads * head_dim * bits / 8
    * (fraction of tokens kept); a quantized cache counts one extra bit per
    number for a 16-bit scale and a 16-bit zero-point per group of 32.
  * MiniKV: Pushing the Limits of LLM Inference via 2-Bit Layer-Discriminative KV
    Cache, §4.4 "KV Cache compression ratio analysis" and §5.2: full cache
    2 * (H * d) * (l_prompt + l_gen) * 2 bytes; H2O 2 * (H * d) * l_prompt *
    (a_HH + a_RW) * 2 bytes; MiniKV (H * d) * (a_HH + a_RW) * l_prompt + (H * d) *
    l_gen bytes (2-bit codes in groups of 16 with an fp16 scale and zero-point:
    8 bytes per 16 numbers).
"""
from __future__ import annotations

from fractions import Fraction


def blog_budget_row(n_layers: int, kv_heads: int, head_dim: int, bits: int,
                    frac=Fraction(1), quantized: bool = False, group: int = 32,
                    meta_bits: int = 32) -> Fraction:
    """Bytes per token of context (exact rational).

    With `quantized`, each number also carries meta_bits / group bits of scale and
    zero-point (16 + 16 bits per group of 32 = 1 bit per number).
    """
    b = Fraction(bits)
    if quantized:
        b += Fraction(meta_bits, group)
    return 2 * n_layers * kv_heads * head_dim * b / 8 * Fraction(frac)


def minikv_sizes(n_layers: int, hidden: int, l_prompt: int, l_gen: int,
                 a_hh=Fraction(1, 4), a_rw=Fraction(1, 4), h2o_budget=Fraction(15, 100)):
    """The §4.4 size formulas, summed over layers (hidden = heads * head_dim).

    Returns dict(full, kivi, h2o, minikv) in bytes (exact rationals).
    """
    hd = n_layers * hidden
    full = 2 * hd * (l_prompt + l_gen) * 2
    kivi = hd * (l_prompt + l_gen)
    h2o = 2 * hd * l_prompt * Fraction(h2o_budget) * 2
    minikv = hd * (Fraction(a_hh) + Fraction(a_rw)) * l_prompt + hd * l_gen
    return {"full": Fraction(full), "kivi": Fraction(kivi), "h2o": Fraction(h2o),
            "minikv": Fraction(minikv)}
