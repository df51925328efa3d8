"""Pins the oracle's full-prompt cumulated attention (MiniKV §4.3 "selective
flash-attention", Figure 9: column sums of the un-normalised FlashAttention
tiles, key blocks visited in order with a running row maximum)."""
import math

import numpy as np
import pytest

from oracle.acumul import acumul_scores, acumul_select


def _hand_case():
    """d = 1, every query 1, keys 0, ln 2, ln 4: S_ij = k_j (scale 1/sqrt(1))."""
    q = np.ones((1, 3, 1))
    k = np.array([[0.0], [math.log(2.0)], [math.log(4.0)]])
    return q, k


@pytest.mark.parametrize("key_block,want", [
    # one key per block: each new key is the row's running maximum, so every
    # visible entry is exp(0) = 1 and A[j] counts the rows i >= j
    (1, [3.0, 2.0, 1.0]),
    # blocks {0, 1}, {2}: row 0 -> A0 += 1; row 1 (max ln2) -> A0 += 1/2, A1 += 1;
    # row 2: first block (max ln2) -> A0 += 1/2, A1 += 1, then key 2 alone -> A2 += 1
    (2, [2.0, 2.0, 1.0]),
    # one block: each row uses its full maximum (row 1: ln2, row 2: ln4)
    # A0 = 1 + 1/2 + 1/4, A1 = 1 + 1/2, A2 = 1
    (3, [1.75, 1.5, 1.0]),
    (128, [1.75, 1.5, 1.0]),
])
def test_hand_computed_example(key_block, want):
    q, k = _hand_case()
    np.testing.assert_allclose(acumul_scores(q, k, key_block), want, rtol=1e-15, atol=0)


@pytest.mark.parametrize("n,g,block", [(1, 1, 128), (200, 1, 128), (300, 3, 64), (129, 2, 128),
                                       (77, 4, 1)])
def test_identical_keys_count_rows(n, g, block):
    """All logits of a row equal: every visible entry is 1, so A[j] = g (n - j)
    whatever the blocking."""
    rng = np.random.default_rng(n)
    q = rng.standard_normal((g, n, 16))
    k = np.tile(rng.standard_normal(16), (n, 1))
    np.testing.assert_allclose(acumul_scores(q, k, block), g * (n - np.arange(n)), rtol=1e-13)


def test_dominant_first_key_makes_blocking_irrelevant():
    """Key 0 carries every row's maximum: the running maximum is final from the
    first block on, so every block size gives the same A_cumul."""
    rng = np.random.default_rng(5)
    n, d, g = 400, 32, 2
    q = rng.standard_normal((g, n, d))
    k = rng.standard_normal((n, d))
    k[0] = 0.0
    q[:, :, 0] = 1.0
    k[0, 0] = 40.0          # logit 40 / sqrt(32) ~ 7 above every other
    k[1:, 0] = 0.0
    ref = acumul_scores(q, k, n)
    for block in (1, 7, 64, 128):
        np.testing.assert_allclose(acumul_scores(q, k, block), ref, rtol=1e-12)


def test_blocked_at_least_unblocked_and_bounded():
    """A running maximum never exceeds the final one, so each blocked entry is at
    least the unblocked one; every entry is at most 1, so A[j] <= g (n - j)."""
    rng = np.random.default_rng(7)
    n, d, g = 513, 64, 2
    q = rng.standard_normal((g, n, d)) * 2.0
    k = rng.standard_normal((n, d))
    full = acumul_scores(q, k, n)
    blk = acumul_scores(q, k, 128)
    assert np.all(blk >= full * (1 - 1e-12))
    assert np.any(blk > full * (1 + 1e-6))          # the blocking does matter here
    assert np.all(blk <= g * (n - np.arange(n)) * (1 + 1e-12))


def test_last_column_and_first_block_of_a_row():
    """Only the last row sees the last key, with its full row maximum:
    A[n-1] = sum_h exp(S_{n-1,n-1} - max_j S_{n-1,j})."""
    rng = np.random.default_rng(9)
    n, d, g = 300, 16, 3
    q = rng.standard_normal((g, n, d))
    k = rng.standard_normal((n, d))
    want = 0.0
    for h in range(g):
        s = k @ q[h, n - 1] / math.sqrt(d)
        want += math.exp(s[n - 1] - s.max())
    assert acumul_scores(q, k, 128)[n - 1] == pytest.approx(want, rel=1e-13)


def test_gqa_heads_add_and_prefix_monotone():
    rng = np.random.default_rng(11)
    n, d = 260, 32
    q = rng.standard_normal((2, n, d))
    k = rng.standard_normal((n, d))
    both = acumul_scores(q, k)
    np.testing.assert_allclose(both, acumul_scores(q[:1], k) + acumul_scores(q[1:], k),
                               rtol=1e-13)
    # a longer prompt only adds rows: A over the first 200 positions can only grow
    short = acumul_scores(q[:, :200], k[:200])
    assert np.all(both[:200] >= short * (1 - 1e-13))


def test_selection_keeps_planted_heavy_hitters():
    """Queries share a direction u (as the synthetic workloads' queries do); keys
    planted along u draw every later row's attention and must be kept."""
    rng = np.random.default_rng(13)
    n, d, g, alpha = 600, 32, 2, 16
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    q = rng.standard_normal((g, n, d)) + 2.0 * u
    k = rng.standard_normal((n, d)) * 0.3
    hitters = [5, 123, 321, 480]
    k[hitters] = 6.0 * u
    idx, s, p = acumul_select(q, k, 32, alpha)
    assert len(s) == n - alpha and np.array_equal(s, p)    # width 1: no pooling
    assert len(idx) == 32 and np.all(np.diff(idx) > 0)
    assert set(hitters) <= set(idx.tolist())


def test_cache_prefill_with_full_prompt_queries():
    """OracleCache keeps, per (sequence, kv head), the A_cumul heavy hitters when
    given every prompt query, and places them as for any selection."""
    from oracle import OracleCache
    rng = np.random.default_rng(17)
    B, Hq, Hk, n, d, alpha = 1, 4, 2, 300, 32, 16
    q = rng.standard_normal((B, Hq, n, d))
    k = rng.standard_normal((B, Hk, n, d))
    v = rng.standard_normal((B, Hk, n, d))
    oc = OracleCache(B, Hq, Hk, d, 2, 32, 64)
    oc.prefill(k, v, alpha, budget=64, q_full=q, pool_kernel=1)
    for h in range(Hk):
        want, _, _ = acumul_select(q[0, 2 * h:2 * h + 2], k[0, h], 64, alpha)
        np.testing.assert_array_equal(oc.heads[0][h].kept, want)
        assert oc.n_packed() == 64 and len(oc.heads[0][h].win_k) == alpha


@pytest.mark.parametrize("n,g,block", [(300, 2, 128), (513, 1, 128), (257, 4, 64), (40, 3, 7)])
def test_sampled_columns_match_the_full_computation(n, g, block):
    """The per-column evaluator (used at full sizes) against the blocked sweep."""
    rng = np.random.default_rng(n + g)
    q = rng.standard_normal((g, n, 32)) * 1.5
    k = rng.standard_normal((n, 32))
    from oracle import acumul_columns
    cols = sorted(set([0, 1, block - 1, block, n // 2, n - 2, n - 1]) & set(range(n)))
    np.testing.assert_allclose(acumul_columns(q, k, cols, block),
                               acumul_scores(q, k, block)[cols], rtol=1e-12)


# ---------------------------------------------------------------- X_O
from oracle.acumul import prefill_attention  # noqa: E402


def test_prefill_attention_identical_keys_is_running_mean():
    """Equal logits in every row: row i averages v_0 .. v_i (a closed form)."""
    rng = np.random.default_rng(5)
    n, d = 40, 8
    q = rng.standard_normal((2, n, d))
    k = np.tile(rng.standard_normal(d), (n, 1))
    v = rng.standard_normal((n, d))
    want = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    got = prefill_attention(q, k, v)
    for h in range(2):
        np.testing.assert_allclose(got[h], want, rtol=1e-13, atol=1e-13)


def test_prefill_attention_two_keys_logistic():
    """Row 1 sees keys 0 and 1 only: its weight on key 1 is the logistic function of
    the logit difference (q.k1 - q.k0)/sqrt(d); row 0 returns v_0 exactly."""
    d = 4
    q = np.zeros((1, 2, d))
    q[0, 1] = [1.0, 2.0, 0.0, 0.0]
    k = np.array([[0.5, 0.0, 0.0, 0.0], [0.0, 1.0, 0.0, 0.0]])
    v = np.array([[1.0, 0.0, 3.0, 0.0], [0.0, 2.0, 0.0, -1.0]])
    got = prefill_attention(q, k, v)
    np.testing.assert_array_equal(got[0, 0], v[0])
    t = (2.0 - 0.5) / math.sqrt(d)
    w1 = 1.0 / (1.0 + math.exp(-t))
    np.testing.assert_allclose(got[0, 1], (1 - w1) * v[0] + w1 * v[1], rtol=1e-14)


def test_prefill_attention_dominant_key_selects_its_value():
    """A key far more aligned with every query than the rest takes (almost) all the
    weight of every row that sees it; rows before it keep their own softmax."""
    rng = np.random.default_rng(6)
    n, d, j = 30, 16, 7
    q = np.abs(rng.standard_normal((1, n, d))) + 1.0
    k = 0.01 * rng.standard_normal((n, d))
    k[j] = 100.0
    v = rng.standard_normal((n, d))
    got = prefill_attention(q, k, v)
    np.testing.assert_allclose(got[0, j:], np.tile(v[j], (n - j, 1)), atol=1e-12)


def test_prefill_attention_is_shift_invariant_per_row():
    """Adding a key-independent vector to every key shifts row i's logits by a
    constant (q_i . c): the output does not change."""
    rng = np.random.default_rng(7)
    n, d = 25, 8
    q = rng.standard_normal((3, n, d))
    k = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    c = rng.standard_normal(d)
    np.testing.assert_allclose(prefill_attention(q, k + c, v), prefill_attention(q, k, v),
                               rtol=1e-12, atol=1e-12)


def test_prefill_attention_last_row_is_dense_decode():
    """The last prompt row attends to every prompt key: it equals one step of plain
    dense attention computed directly (the special case the cache must reach with
    the full budget and 16-bit storage)."""
    rng = np.random.default_rng(8)
    n, d = 33, 8
    q = rng.standard_normal((1, n, d))
    k = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    s = k @ q[0, -1] / math.sqrt(d)
    w = np.exp(s - s.max())
    np.testing.assert_allclose(prefill_attention(q, k, v)[0, -1], (w / w.sum()) @ v, rtol=1e-13)
