"""Pins the oracle's compressed cache: dense equivalence, window schedule, FIFO flush."""
import numpy as np
import pytest
import torch

import synth
from oracle import OracleCache, quantize_keys, quantize_values


def _sdpa(q, K, V):
    """Library dense attention (one query row, all keys visible), float64."""
    qt = torch.from_numpy(q)[None, None, None]          # [1,1,1,d]
    out = torch.nn.functional.scaled_dot_product_attention(
        qt, torch.from_numpy(K)[None, None], torch.from_numpy(V)[None, None])
    return out[0, 0, 0].numpy()


@pytest.mark.parametrize("gqa,alpha", [(1, 8), (4, 0), (2, 16)])
def test_full_budget_16bit_is_dense_attention(gqa, alpha):
    """budget = prompt length and 16-bit storage: decode == plain dense attention."""
    spec = synth.small_spec(2, n_layers=1, batch=2, n_q_heads=2 * gqa, n_kv_heads=2,
                            head_dim=32, prompt_len=200, obs_window=alpha, window_len=64,
                            bits=16)
    x = synth.layer_inputs(spec, 0)
    k, v = x["k"].double().numpy(), x["v"].double().numpy()
    cache = OracleCache(2, 2 * gqa, 2, 32, 16, 32, 64)
    cache.prefill(k, v, alpha, budget=None)
    K_all, V_all = list(k), list(v)
    K_all = [[k[b, h] for h in range(2)] for b in range(2)]
    V_all = [[v[b, h] for h in range(2)] for b in range(2)]
    for t in range(70):                     # crosses two flushes
        dx = synth.decode_inputs(spec, 0, t)
        q = dx["q"].double().numpy()
        kn, vn = dx["k_new"].double().numpy(), dx["v_new"].double().numpy()
        o = cache.step(q, kn, vn)
        for b in range(2):
            for h in range(2):
                K_all[b][h] = np.vstack([K_all[b][h], kn[b, h][None]])
                V_all[b][h] = np.vstack([V_all[b][h], vn[b, h][None]])
            for hq in range(2 * gqa):
                ref = _sdpa(q[b, hq], K_all[b][hq // gqa], V_all[b][hq // gqa])
                np.testing.assert_allclose(o[b, hq], ref, rtol=1e-12, atol=1e-12)


def test_window_schedule_closed_form():
    """Window length after t appends: w0 + t minus G per flush, a flush whenever the
    length reaches R; the packed store grows by G per flush."""
    for (w0, R, G, k0) in [(16, 32, 32, 128), (32, 128, 32, 512), (0, 128, 32, 1024),
                           (32, 64, 32, 128)]:
        cache = OracleCache(1, 1, 1, 32, 2, G, R)
        n = k0 + w0
        rng = np.random.default_rng(0)
        kk = rng.normal(size=(1, 1, n, 32)).astype(np.float32).astype(np.float64)
        cache.prefill(kk, kk, w0, budget=None)
        assert cache.window_len() == w0 and cache.n_packed() == k0
        flushes = 0
        for t in range(1, 300):
            cache.append(rng.normal(size=(1, 1, 32)), rng.normal(size=(1, 1, 32)))
            if w0 + t - G * flushes == R:
                flushes += 1
            assert cache.window_len() == w0 + t - G * flushes
            assert cache.n_packed() == k0 + G * flushes
            assert cache.window_len() < R


def test_flush_takes_the_oldest_group():
    """The group quantized at a flush is exactly the G oldest window tokens."""
    G, R, d = 32, 64, 64
    rng = np.random.default_rng(1)
    n, a = 96, 32
    k = rng.normal(size=(1, 1, n, d)).astype(np.float32).astype(np.float64)
    v = rng.normal(size=(1, 1, n, d)).astype(np.float32).astype(np.float64)
    cache = OracleCache(1, 1, 1, d, 2, G, R)
    cache.prefill(k, v, a, budget=None)
    news_k, news_v = [], []
    for t in range(R - a):
        nk = rng.normal(size=(1, 1, d)).astype(np.float32).astype(np.float64)
        nv = rng.normal(size=(1, 1, d)).astype(np.float32).astype(np.float64)
        news_k.append(nk[0, 0]); news_v.append(nv[0, 0])
        cache.append(nk, nv)
    st = cache.heads[0][0]
    # after the flush: packed = 64 prompt tokens + the 32 observation tokens
    oldest_k = k[0, 0, n - a:]
    kc, kS, kZ = quantize_keys(oldest_k, 2, G)
    np.testing.assert_array_equal(st.kcodes[-G:], kc)
    np.testing.assert_array_equal(st.kS[-1:], kS)
    vc, vS, vZ = quantize_values(v[0, 0, n - a:], 2, G)
    np.testing.assert_array_equal(st.vcodes[-G:], vc)
    np.testing.assert_array_equal(st.win_k, np.array(news_k))


def test_selected_tail_goes_to_window():
    """Kept tokens past the last whole group start the bf16 window, before the
    observation tokens."""
    rng = np.random.default_rng(2)
    n, d, a, G = 120, 32, 8, 32
    k = rng.normal(size=(1, 1, n, d)).astype(np.float32).astype(np.float64)
    cache = OracleCache(1, 1, 1, d, 2, G, 64)
    kept = [[np.array(sorted(rng.choice(n - a, 40, replace=False)))]]
    cache.prefill(k, k, a, kept=kept)
    st = cache.heads[0][0]
    assert st.n_packed == 32
    np.testing.assert_array_equal(st.win_k[:8], k[0, 0, kept[0][0][32:]])
    np.testing.assert_array_equal(st.win_k[8:], k[0, 0, n - a:])


def test_flush_all_agrees_when_window_equals_group():
    """MiniKV (Algorithm 1, decoding) keeps new tokens in a 16-bit buffer and, when
    it holds n_r tokens, quantizes all of them and empties it; the cache here flushes
    its oldest group whenever the window reaches R. With R = G = n_r the two are the
    same schedule: restated independently below (a list that is quantized whole and
    cleared), the packed store and the window agree after every step."""
    G = R = 32
    d, n, a = 32, 200, 16
    rng = np.random.default_rng(3)
    k = rng.normal(size=(1, 1, n, d)).astype(np.float32).astype(np.float64)
    v = rng.normal(size=(1, 1, n, d)).astype(np.float32).astype(np.float64)
    cache = OracleCache(1, 1, 1, d, 2, G, R)
    kept = [[np.arange(0, 2 * G)]]                 # two whole groups, no tail
    cache.prefill(k, v, a, kept=kept)
    st = cache.heads[0][0]
    # flush-all model: the buffer starts with the observation tokens
    buf_k, buf_v = list(k[0, 0, n - a:]), list(v[0, 0, n - a:])
    packed_k = [st.kcodes.copy()]
    for t in range(100):
        nk = rng.normal(size=(1, 1, d)).astype(np.float32).astype(np.float64)
        nv = rng.normal(size=(1, 1, d)).astype(np.float32).astype(np.float64)
        cache.append(nk, nv)
        buf_k.append(nk[0, 0])
        buf_v.append(nv[0, 0])
        if len(buf_k) == R:                        # n_r tokens: quantize all, empty
            kc, kS, kZ = quantize_keys(np.array(buf_k), 2, G)
            vc, vS, vZ = quantize_values(np.array(buf_v), 2, G)
            packed_k.append(kc)
            np.testing.assert_array_equal(st.kcodes[-G:], kc)
            np.testing.assert_array_equal(st.vcodes[-G:], vc)
            np.testing.assert_array_equal(st.kS[-1:], kS)
            np.testing.assert_array_equal(st.vS[-G:], vS)
            buf_k, buf_v = [], []
        np.testing.assert_array_equal(st.kcodes, np.vstack(packed_k))
        assert len(st.win_k) == len(buf_k)
        if buf_k:
            np.testing.assert_array_equal(st.win_k, np.array(buf_k))
            np.testing.assert_array_equal(st.win_v, np.array(buf_v))
