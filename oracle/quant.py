"""KIVI-style asymmetric group quantization -- oracle (test infrastructure only).

Follows:
  * KV Cache Compression: Eviction and Quantization (blog), "Quantization: keep
    each token in fewer bits" and "Measured on a real model": every group has a
    zero-point equal to the group minimum and a scale (max - min) / (2^b - 1);
    values are rounded to the nearest level; keys are grouped per channel (one
    channel over a group of tokens), values per token (one token over a group of
    channels); "The budget" counts a 16-bit scale and a 16-bit zero-point per
    group of 32 numbers.
  * MiniKV: Pushing the Limits of LLM Inference via 2-Bit Layer-Discriminative KV
    Cache, §4.4: the selected keys/values are quantized along the channel / token
    dimension respectively, codes packed into INT32 words, zero-point and scale
    stored as FP16.

Arithmetic (the order of operations is a reading; the pages leave it open):
  all in IEEE fp32 with round-to-nearest-even and no fused multiply-add --
    lo = min(x), hi = max(x), s32 = (hi - lo) / (2^b - 1)   [true division],
    S = fp16(s32), Z = fp16(lo)                              [round-to-nearest-even],
    code = rint((x - float(Z)) / float(S)), clamped to [0, 2^b - 1]
           (rint = round half to even; the stored fp16 values are used so that
            dequantization code * S + Z reproduces the stored state exactly),
    S == 0 (constant group, or a scale below fp16's range) gives all-zero codes.
  dequantized value: code * S + Z (evaluated exactly, in fp64).
"""
from __future__ import annotations

import numpy as np


def _quantize_along(x: np.ndarray, axis: int, bits: int):
    """Quantize groups that run along `axis` of a float32 array.

    Returns (codes uint8 same shape as x, S fp16, Z fp16) with S/Z keeping `axis`
    as a length-1 dimension.
    """
    if bits not in (2, 4, 8):
        raise ValueError("bits must be 2, 4 or 8")
    x32 = np.asarray(x, dtype=np.float32)
    levels = np.float32(2 ** bits - 1)
    lo = x32.min(axis=axis, keepdims=True)
    hi = x32.max(axis=axis, keepdims=True)
    rng = (hi - lo).astype(np.float32)              # fp32 subtraction
    s32 = (rng / levels).astype(np.float32)         # fp32 IEEE division
    S = s32.astype(np.float16)                      # round-to-nearest-even
    Z = lo.astype(np.float16)
    Sf = S.astype(np.float32)
    Zf = Z.astype(np.float32)
    diff = (x32 - Zf).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (diff / Sf).astype(np.float32)
    codes = np.rint(q)                              # half to even
    codes = np.where(Sf == 0, np.float32(0), codes)
    codes = np.clip(codes, 0, levels).astype(np.uint8)
    return codes, S, Z


def quantize_group(x: np.ndarray, bits: int):
    """Quantize one group (1-D). Returns (codes uint8 [n], S fp16 scalar, Z fp16 scalar)."""
    codes, S, Z = _quantize_along(np.asarray(x, np.float32).reshape(1, -1), 1, bits)
    return codes[0], S[0, 0], Z[0, 0]


def quantize_keys(k: np.ndarray, bits: int, group: int):
    """Per-channel key quantization over groups of `group` consecutive tokens.

    k: [T][d] with T a multiple of `group`. Returns codes [T][d] uint8,
    S, Z [T/group][d] fp16.
    """
    T, d = k.shape
    if T % group:
        raise ValueError("token count must be a multiple of the group size")
    codes, S, Z = _quantize_along(np.asarray(k, np.float32).reshape(T // group, group, d),
                                  1, bits)
    return codes.reshape(T, d), S[:, 0, :], Z[:, 0, :]


def quantize_values(v: np.ndarray, bits: int, group: int):
    """Per-token value quantization over groups of `group` consecutive channels.

    v: [T][d] with d a multiple of `group`. Returns codes [T][d] uint8,
    S, Z [T][d/group] fp16.
    """
    T, d = v.shape
    if d % group:
        raise ValueError("head_dim must be a multiple of the group size")
    codes, S, Z = _quantize_along(np.asarray(v, np.float32).reshape(T, d // group, group),
                                  2, bits)
    return codes.reshape(T, d), S[:, :, 0], Z[:, :, 0]


def dequantize_keys(codes: np.ndarray, S: np.ndarray, Z: np.ndarray, group: int):
    """codes [T][d], S/Z [T/group][d] -> fp64 [T][d]."""
    Sg = np.repeat(S.astype(np.float64), group, axis=0)
    Zg = np.repeat(Z.astype(np.float64), group, axis=0)
    return codes.astype(np.float64) * Sg + Zg


def dequantize_values(codes: np.ndarray, S: np.ndarray, Z: np.ndarray, group: int):
    """codes [T][d], S/Z [T][d/group] -> fp64 [T][d]."""
    Sg = np.repeat(S.astype(np.float64), group, axis=1)
    Zg = np.repeat(Z.astype(np.float64), group, axis=1)
    return codes.astype(np.float64) * Sg + Zg
