"""The compressed KV cache of one layer -- oracle (test infrastructure only).

Follows:
  * MiniKV: Pushing the Limits of LLM Inference via 2-Bit Layer-Discriminative KV
    Cache, §4.1 (the set selected at the end of prefill is quantized once and
    frozen), §4.4 and Algorithm 1: prefill keeps the selected tokens and
    quantizes them (keys per channel, values per token); every decode step
    appends the new key/value to a 16-bit streaming buffer, quantizes the buffer
    when it fills, and attends with one softmax over the concatenation of the
    dequantized keys and the buffer's keys; the output is
    A_quant . dequant(Q_V) + A_unquant . R_V.
  * KV Cache Compression: Eviction and Quantization (blog), "Quantization: keep
    each token in fewer bits" and "Measured on a real model": recent tokens stay
    in full precision until a group fills; attention reads the exact keys/values
    of the recent window and the rounded ones of everything else, one softmax over
    both.
  * PyramidKV: Dynamic KV Cache Compression based on Pyramidal Information
    Funneling, §4.2: the last alpha prompt tokens are always kept.

Readings:
  * The packed store holds whole groups of G kept tokens in ascending position
    order. The kept tokens past the last whole group (k mod G of them) and then
    the alpha observation tokens start the bf16 window (with no eviction, alpha = 0
    and the window starts with the last n mod G prompt tokens).
  * The window is flushed group by group: after an append, when its length
    reaches R, its oldest G tokens are quantized as one new key group and G value
    rows and leave the window. (MiniKV flushes the whole buffer every n_r steps;
    the two agree when R == G.)
  * bits == 16 stores the selected tokens exactly (no quantization): the special
    case in which the method must reduce to dense attention.
"""
from __future__ import annotations

import math
from typing import List, Optional

import numpy as np

from .quant import quantize_keys, quantize_values, dequantize_keys, dequantize_values
from .acumul import acumul_select
from .snapkv import snapkv_select


class _Head:
    """State of one (sequence, kv head)."""

    def __init__(self, d: int, group: int, bits: int):
        self.d, self.G, self.bits = d, group, bits
        self.kept = np.zeros(0, dtype=np.int64)
        self.kcodes = np.zeros((0, d), np.uint8)
        self.kS = np.zeros((0, d), np.float16)
        self.kZ = np.zeros((0, d), np.float16)
        self.vcodes = np.zeros((0, d), np.uint8)
        self.vS = np.zeros((0, d // group), np.float16)
        self.vZ = np.zeros((0, d // group), np.float16)
        self.k_hat = np.zeros((0, d))       # dequantized packed keys (fp64)
        self.v_hat = np.zeros((0, d))
        self.win_k = np.zeros((0, d))       # bf16 window, oldest first (exact values)
        self.win_v = np.zeros((0, d))

    def pack(self, k_rows: np.ndarray, v_rows: np.ndarray):
        """Quantize whole groups of rows and append them to the packed store."""
        if len(k_rows) == 0:
            return
        if self.bits == 16:
            self.k_hat = np.vstack([self.k_hat, k_rows])
            self.v_hat = np.vstack([self.v_hat, v_rows])
            return
        kc, kS, kZ = quantize_keys(k_rows, self.bits, self.G)
        vc, vS, vZ = quantize_values(v_rows, self.bits, self.G)
        self.kcodes = np.vstack([self.kcodes, kc])
        self.kS = np.vstack([self.kS, kS])
        self.kZ = np.vstack([self.kZ, kZ])
        self.vcodes = np.vstack([self.vcodes, vc])
        self.vS = np.vstack([self.vS, vS])
        self.vZ = np.vstack([self.vZ, vZ])
        self.k_hat = np.vstack([self.k_hat, dequantize_keys(kc, kS, kZ, self.G)])
        self.v_hat = np.vstack([self.v_hat, dequantize_values(vc, vS, vZ, self.G)])

    @property
    def n_packed(self) -> int:
        return len(self.k_hat)


class OracleCache:
    """Compressed cache of one layer for B sequences x Hkv kv heads."""

    def __init__(self, batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                 bits: int, group: int, window_len: int):
        if n_q_heads % n_kv_heads:
            raise ValueError("n_q_heads must be a multiple of n_kv_heads")
        if window_len < group or window_len % group:
            raise ValueError("window_len must be a positive multiple of the group size")
        self.B, self.Hq, self.Hk, self.d = batch, n_q_heads, n_kv_heads, head_dim
        self.gqa = n_q_heads // n_kv_heads
        self.bits, self.G, self.R = bits, group, window_len
        self.heads = [[_Head(head_dim, group, bits) for _ in range(n_kv_heads)]
                      for _ in range(batch)]
        self.scores = None      # [B][Hk] arrays of s (selection scores) when scored
        self.pooled = None

    # ------------------------------------------------------------------ prefill
    def prefill(self, k: np.ndarray, v: np.ndarray, obs_window: int,
                budget: Optional[int] = None, q_obs: Optional[np.ndarray] = None,
                pool_kernel: int = 7, kept: Optional[List[List[np.ndarray]]] = None,
                q_full: Optional[np.ndarray] = None):
        """Select, quantize and place the prompt.

        k, v: [B][Hkv][n][d] (exact bf16 values). q_obs: [B][Hq][alpha][d].
        Selection: `kept` if given (ascending indices in [0, n - alpha) per (b, h)),
        else the top-`budget` when budget < n - alpha -- of the full-prompt
        cumulated attention when `q_full` ([B][Hq][n][d], every prompt query) is
        given, else of the observation-window score -- else all.
        """
        B, Hk, n, d = k.shape
        a = obs_window
        if a >= n:
            raise ValueError("observation window must be shorter than the prompt")
        self.scores = [[None] * Hk for _ in range(B)]
        self.pooled = [[None] * Hk for _ in range(B)]
        for b in range(B):
            for h in range(Hk):
                if kept is not None:
                    idx = np.asarray(kept[b][h], dtype=np.int64)
                elif budget is not None and budget < n - a and q_full is not None:
                    qg = q_full[b, h * self.gqa:(h + 1) * self.gqa].astype(np.float64)
                    idx, s, p = acumul_select(qg, k[b, h].astype(np.float64), budget, a,
                                              pool_kernel)
                    self.scores[b][h], self.pooled[b][h] = s, p
                elif budget is not None and budget < n - a:
                    if q_obs is None:
                        raise ValueError("scoring needs the observation queries")
                    qg = q_obs[b, h * self.gqa:(h + 1) * self.gqa].astype(np.float64)
                    idx, s, p = snapkv_select(qg, k[b, h].astype(np.float64), budget,
                                              pool_kernel)
                    self.scores[b][h], self.pooled[b][h] = s, p
                else:
                    idx = np.arange(n - a, dtype=np.int64)
                st = self.heads[b][h]
                st.kept = idx
                full = (len(idx) // self.G) * self.G
                kk = k[b, h].astype(np.float64)
                vv = v[b, h].astype(np.float64)
                st.pack(kk[idx[:full]], vv[idx[:full]])
                tail = np.concatenate([idx[full:], np.arange(n - a, n)]).astype(np.int64)
                st.win_k = kk[tail].copy()
                st.win_v = vv[tail].copy()
                if len(tail) >= self.R:
                    raise ValueError("initial window must be shorter than window_len")

    # ------------------------------------------------------------------- decode
    def append(self, k_new: np.ndarray, v_new: np.ndarray):
        """Append one token per (b, h) (k_new, v_new: [B][Hkv][d]); flush a full window."""
        for b in range(self.B):
            for h in range(self.Hk):
                st = self.heads[b][h]
                st.win_k = np.vstack([st.win_k, k_new[b, h].astype(np.float64)[None]])
                st.win_v = np.vstack([st.win_v, v_new[b, h].astype(np.float64)[None]])
                if len(st.win_k) == self.R:
                    st.pack(st.win_k[:self.G], st.win_v[:self.G])
                    st.win_k = st.win_k[self.G:]
                    st.win_v = st.win_v[self.G:]

    def attend(self, q: np.ndarray) -> np.ndarray:
        """Decode attention of one query per head (q: [B][Hq][d]) -> o [B][Hq][d] fp64."""
        o = np.zeros((self.B, self.Hq, self.d))
        scale = 1.0 / math.sqrt(self.d)
        for b in range(self.B):
            for hq in range(self.Hq):
                st = self.heads[b][hq // self.gqa]
                keys = np.vstack([st.k_hat, st.win_k])
                vals = np.vstack([st.v_hat, st.win_v])
                logits = keys @ q[b, hq].astype(np.float64) * scale
                w = np.exp(logits - logits.max())
                o[b, hq] = (w / w.sum()) @ vals
        return o

    def step(self, q, k_new, v_new) -> np.ndarray:
        """One decode step: append then attend."""
        self.append(k_new, v_new)
        return self.attend(q)

    # ---------------------------------------------------------------- inspection
    def window_len(self) -> int:
        return len(self.heads[0][0].win_k)

    def n_packed(self) -> int:
        return self.heads[0][0].n_packed
