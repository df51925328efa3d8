"""Pins the oracle's KIVI-style group quantizer."""
import struct

import numpy as np
import pytest

from oracle import (quantize_group, quantize_keys, quantize_values, dequantize_keys,
                    dequantize_values)


def _bf16(x):
    """Round fp64 values to bf16 (nearest even) and return them as fp32."""
    import torch
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def _half_rne_bits(f32):
    """IEEE binary16 round-to-nearest-even of a normal-range float32, from the
    definition (not numpy): keep 10 fraction bits, round on the dropped 13."""
    u = struct.unpack("<I", struct.pack("<f", float(f32)))[0]
    sign, exp, frac = u >> 31, (u >> 23) & 0xFF, u & 0x7FFFFF
    e = exp - 127 + 15
    assert 1 <= e <= 30
    mant = frac >> 13
    rest = frac & 0x1FFF
    if rest > 0x1000 or (rest == 0x1000 and (mant & 1)):
        mant += 1
        if mant == 1024:
            mant, e = 0, e + 1
    return (sign << 15) | (e << 10) | mant


def test_fp16_rounding_is_nearest_even():
    """The oracle relies on numpy's float32 -> float16 being IEEE RNE; check ties."""
    rng = np.random.default_rng(0)
    vals = list(rng.normal(size=2000).astype(np.float32) * 7)
    for m in range(0, 1024, 37):            # exact halfway cases at several exponents
        for e in (-3, 0, 5):
            base = (1 + m / 1024) * 2.0 ** e
            vals.append(np.float32(base + 2.0 ** (e - 11)))
            vals.append(np.float32(-(base + 2.0 ** (e - 11))))
    for v in vals:
        assert int(np.float32(v).astype(np.float16).view(np.uint16)) == _half_rne_bits(v)


@pytest.mark.parametrize("bits", [2, 4])
def test_codes_are_nearest_levels(bits):
    rng = np.random.default_rng(bits)
    for trial in range(200):
        x = _bf16(rng.normal(size=32) * rng.lognormal(0, 1) + rng.normal())
        c, S, Z = quantize_group(x, bits)
        Sf, Zf = float(S), float(Z)
        assert c.max() <= 2 ** bits - 1
        levels = np.arange(2 ** bits) * Sf + Zf
        err = np.abs(x[:, None].astype(np.float64) - levels[None, :])
        chosen = err[np.arange(32), c]
        # nearest level (up to one fp32 rounding of (x - Z) / S)
        assert (chosen <= err.min(axis=1) + 1e-6 * Sf).all()
        # dequantization error within half a step for elements inside the grid
        inside = (x >= Zf) & (x <= Zf + (2 ** bits - 1) * Sf)
        assert (np.abs(x - (c * Sf + Zf))[inside] <= 0.5 * Sf * (1 + 2 ** -20)).all()


@pytest.mark.parametrize("bits", [2, 4])
def test_scale_and_zero(bits):
    x = np.array([-1.5, 0.25, 2.0, 0.0] * 8, np.float32)
    c, S, Z = quantize_group(x, bits)
    assert np.float16(Z) == np.float16(-1.5)
    assert S == np.float16(np.float32(np.float32(3.5) / np.float32(2 ** bits - 1)))
    assert c[0] == 0 and c[2] == 2 ** bits - 1


def test_round_half_to_even():
    """(x - Z) / S exactly k + 1/2 rounds to the even code."""
    x = np.array([0.0, 3.0, 0.5, 1.5, 2.5] + [0.0] * 27, np.float32)
    c, S, Z = quantize_group(x, 2)
    assert float(S) == 1.0 and float(Z) == 0.0
    assert list(c[:5]) == [0, 3, 0, 2, 2]


def test_constant_group():
    x = np.full(32, 0.7, np.float32)
    c, S, Z = quantize_group(x, 2)
    assert float(S) == 0.0 and (c == 0).all() and Z == np.float16(0.7)


def test_key_groups_run_along_tokens():
    """Per-channel keys: a channel constant over its 32 tokens is stored exactly
    even when channels differ wildly; per-token values: a token constant over its
    32 channels is stored exactly."""
    rng = np.random.default_rng(7)
    T, d, G = 64, 64, 32
    chan = _bf16(rng.normal(size=d) * 100)
    k = np.repeat(np.tile(chan, (G, 1)), T // G, axis=0)
    kc, kS, kZ = quantize_keys(k, 2, G)
    assert kS.shape == (T // G, d) and (kS == 0).all()
    np.testing.assert_array_equal(dequantize_keys(kc, kS, kZ, G),
                                  np.float16(k).astype(np.float64))
    tok = _bf16(rng.normal(size=T) * 100)
    v = np.tile(tok[:, None], (1, d))
    vc, vS, vZ = quantize_values(v, 2, G)
    assert vS.shape == (T, d // G) and (vS == 0).all()
    # a per-token layout of the keys would not be exact
    kc2, kS2, kZ2 = quantize_values(k, 2, G)
    assert (kS2 != 0).any()


def test_dequant_error_bound_on_workload_distribution():
    """|x - xhat| <= S/2 on keys with LogNormal channel scales; count clamps."""
    rng = np.random.default_rng(8)
    T, d, G = 256, 128, 32
    k = _bf16(rng.normal(size=(T, d)) * np.exp(rng.normal(size=d) * 0.5))
    for bits in (2, 4):
        kc, kS, kZ = quantize_keys(k, bits, G)
        kh = dequantize_keys(kc, kS, kZ, G)
        Sg = np.repeat(kS.astype(np.float64), G, axis=0)
        err = np.abs(k - kh)
        over = err > 0.5 * Sg * (1 + 2 ** -20)
        # elements outside the fp16-rounded grid (clamped) are the only exceptions
        assert over.sum() <= 0.01 * over.size
        vc, vS, vZ = quantize_values(k, bits, G)
        vh = dequantize_values(vc, vS, vZ, G)
        Sv = np.repeat(vS.astype(np.float64), G, axis=1)
        assert (np.abs(k - vh) > 0.5 * Sv * (1 + 2 ** -20)).sum() <= 0.01 * k.size
