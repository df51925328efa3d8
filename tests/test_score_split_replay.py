"""A CPU replay of the scoring launch's work decomposition (index arithmetic
only), checking the invariants its cross-CTA waits and its statistics scratch
rest on:

  * `owner_of` is the inverse of `slice_of`: item i lies in the slice of the CTA
    it names, for every item of every decomposition replayed;
  * the grid never exceeds the row-statistics items, so every CTA owns at least
    one (and the launch's arrival count is reached);
  * the row-statistics tiles of a unit are held by a contiguous run of CTAs
    [cf, cl]; each writes one partial per row into slot (cta - cf) of the unit,
    which stays below the scratch's slots per unit (smax), and counts itself in
    once;
  * a CTA's column phase waits for exactly cl - cf + 1 arrivals, the number that
    come, and reads exactly the slots written; every column item is processed by
    one CTA;
  * `next_unit`, which decides when a CTA's query buffer changes hands, names the
    unit of the item that really comes next in the CTA's walk.

The decomposition restated here is the one of the scoring kernel (score_tc.cu:
`slice_of`, `owner_of`, `next_unit`, the row-statistics and column phases, and the
launch's grid), with 256-key tiles and the scratch sized as in cache creation
(score_stat_chunks: 4 * ceil(n / 128) + 4 slots per unit)."""
import random

import pytest

KEYS = 256


def slice_of(total, c, G):
    return total * c // G, total * (c + 1) // G


def owner_of(i, total, G):
    return ((i + 1) * G + total - 1) // total - 1


def next_unit(ubatch, units, tiles0, tiles1, G, cta, nbatch, j, ph, i):
    while True:
        u0, nu = j * ubatch, min(ubatch, units - j * ubatch)
        tiles = tiles1 if ph else tiles0
        b, e = slice_of(nu * tiles, cta, G)
        if i + 1 < e:
            return u0 + (i + 1) // tiles
        if ph == 0:
            ph = 1
        else:
            ph = 0
            j += 1
            if j >= nbatch:
                return -1
        v0, nv = j * ubatch, min(ubatch, units - j * ubatch)
        i = slice_of(nv * (tiles1 if ph else tiles0), cta, G)[0] - 1


def replay(units, n, alpha, max_ctas, ubatch=None):
    tiles0 = (n + KEYS - 1) // KEYS
    tiles1 = (n - alpha + KEYS - 1) // KEYS
    smax = 4 * ((n + 127) // 128) + 4
    ubatch = units if ubatch is None else ubatch
    items0 = min(ubatch, units) * tiles0
    G = min(max_ctas, items0)
    assert G >= 1
    nbatch = (units + ubatch - 1) // ubatch
    slots = {}                       # (unit, slot) -> cta
    arrivals = {}
    walk = {c: [] for c in range(G)}
    col_done = set()
    for j in range(nbatch):
        u0, nu = j * ubatch, min(ubatch, units - j * ubatch)
        tot0, tot1 = nu * tiles0, nu * tiles1
        # the batched form's precondition: every CTA holds a row-statistics tile of
        # every batch (a unit's wait counts the CTAs over its tiles)
        assert tot0 >= G, "a batch with fewer row items than CTAs"
        # every item's owner is the CTA whose slice holds it
        for total in (tot0, tot1):
            for i in (range(total) if total <= 4096 else random.Random(total).sample(range(total), 4096)):
                o = owner_of(i, total, G)
                b, e = slice_of(total, o, G)
                assert 0 <= o < G and b <= i < e
        # row-statistics phase
        for cta in range(G):
            b, e = slice_of(tot0, cta, G)
            assert e > b, "every CTA owns a row-statistics item of the batch"
            i = b
            while i < e:
                ul = i // tiles0
                iend = min(e, (ul + 1) * tiles0)
                for ii in range(i, iend):
                    walk[cta].append((j, 0, ii, u0 + ii // tiles0))
                i = iend
                cf = owner_of(ul * tiles0, tot0, G)
                slot = cta - cf
                assert 0 <= slot < smax, "partial slot inside the scratch"
                assert (u0 + ul, slot) not in slots, "a partial slot written twice"
                slots[(u0 + ul, slot)] = cta
                arrivals[u0 + ul] = arrivals.get(u0 + ul, 0) + 1
        # column phase
        for cta in range(G):
            b, e = slice_of(tot1, cta, G)
            cur = -1
            for i in range(b, e):
                ul, tile = i // tiles1, i % tiles1
                walk[cta].append((j, 1, i, u0 + ul))
                assert (u0 + ul, tile) not in col_done
                col_done.add((u0 + ul, tile))
                if ul != cur:
                    cur = ul
                    cf = owner_of(ul * tiles0, tot0, G)
                    cl = owner_of((ul + 1) * tiles0 - 1, tot0, G)
                    nct = cl - cf + 1
                    assert arrivals[u0 + ul] == nct, "the wait target is the arrival count"
                    assert all(slots.get((u0 + ul, s)) == cf + s for s in range(nct)), \
                        "the merge reads the slots the unit's CTAs wrote"
                    assert nct <= tiles0 <= smax
    assert len(col_done) == units * tiles1, "every column item processed"
    assert set(arrivals) == set(range(units))
    # next_unit against the walk each CTA really takes
    for cta, items in walk.items():
        for k, (j, ph, i, u) in enumerate(items):
            want = items[k + 1][3] if k + 1 < len(items) else -1
            assert next_unit(ubatch, units, tiles0, tiles1, G, cta, nbatch, j, ph, i) == want
    return G


def test_workload_shapes():
    """The benchmark's workloads at 152 resident CTAs: long context (8 units,
    131,072 keys, 64 observation rows), Llama-3-8B (8 units, 32,768 keys), the
    batched one (128 units, 8,192 keys)."""
    assert replay(8, 131072, 64, 152) == 152
    assert replay(8, 32768, 32, 152) == 152
    assert replay(128, 8192, 32, 152) == 152


@pytest.mark.parametrize("seed", range(4))
def test_random_shapes(seed):
    rng = random.Random(seed)
    for _ in range(150):
        units = rng.choice([1, 2, 3, 8, 16, 33])
        n = rng.choice([2, 17, 255, 256, 257, 600, 1000, 4096, 5000, rng.randint(2, 20000)])
        alpha = rng.randint(1, min(n - 1, 256))
        replay(units, n, alpha, rng.choice([1, 2, 5, 148, 152, 304]))


def test_batched_walks():
    """The kernel's batched form (it launches one batch today): the walk, the
    slots and the wait targets hold for every batch size that gives each CTA a
    row-statistics tile of every batch; a smaller last batch breaks that
    precondition, which the replay detects."""
    rng = random.Random(7)
    checked = 0
    for _ in range(200):
        units = rng.choice([3, 8, 17])
        n = rng.choice([300, 1000, 3000])
        alpha, max_ctas, ub = rng.randint(1, 64), rng.choice([2, 7, 152]), rng.randint(1, units)
        tiles0 = (n + KEYS - 1) // KEYS
        G = min(max_ctas, min(ub, units) * tiles0)
        last = units - (units - 1) // ub * ub
        if last * tiles0 >= G:
            replay(units, n, alpha, max_ctas, ubatch=ub)
            checked += 1
        else:
            with pytest.raises(AssertionError, match="fewer row items than CTAs"):
                replay(units, n, alpha, max_ctas, ubatch=ub)
    assert checked > 50


def test_degenerate_shapes():
    assert replay(1, 2, 1, 152) == 1            # one key tile, one CTA
    assert replay(1, 256, 255, 152) == 1
    assert replay(1, 257, 1, 152) == 2          # two tiles over two CTAs
    assert replay(8192, 300, 16, 152) == 152    # more units than CTAs
