"""A CPU replay of the decode launch's work decomposition (index arithmetic
only; no attention arithmetic), over many random layouts of layers, units and
grid sizes, checking the invariants the kernel's correctness and memory safety
rest on:

  * the launch's chunk list (every layer's units, window chunks then packed
    chunks) is cut into one contiguous range per CTA and each CTA's range into
    one contiguous range per warp: every chunk is processed by exactly one warp;
  * a warp's cursor (layer, unit, chunk) advanced chunk by chunk agrees with a
    direct lookup, and its segments (runs of one unit) are numbered as the
    kernel numbers them;
  * every unit with stored tokens is written exactly once: by the warp holding
    it whole, by the last of a CTA's holders (shared-memory ticket), or by the
    last CTA holding it (global ticket);
  * every partial state goes to a slot (two per warp in shared memory, two per
    CTA in global memory) that nothing else writes in the launch, and each merge
    reads exactly the slots its holders wrote;
  * every ticket counts exactly the arrivals its last arriver waits for, and is
    back at zero when the launch ends;
  * the 32-bit form of the even split is used only where its products fit.

The decomposition restated here is the one of the decode kernel (decode.cu:
`Split`, `locate`/`step`, `finish`); the layouts include empty layers, units of
one chunk, more warps than chunks and grids of 1 to 152 CTAs."""
import random

import pytest


class Split:
    """[base, base + T) cut into N contiguous ranges."""

    def __init__(self, T, N, base):
        self.T, self.N, self.base = T, N, base

    def first(self, i):
        if self.T * self.N < (1 << 32):
            # 32-bit form: i <= N, so i * T <= N * T < 2^32
            assert 0 <= i <= self.N and i * self.T < (1 << 32)
        return self.base + i * self.T // self.N

    def owner(self, c):
        x = c - self.base
        assert 0 <= x < self.T
        if self.T * self.N < (1 << 32):
            assert (x + 1) * self.N < (1 << 32)
        return ((x + 1) * self.N - 1) // self.T


def replay(layers, units, NW, n_sm):
    """layers: [(wchunks, pchunks)] per layer of the launch. Returns the number of
    CTAs, after checking every invariant."""
    begins, total = [], 0
    for w, p in layers:
        begins.append(total)
        total += units * (w + p)
    if total == 0:
        return 0     # the host writes zeros and launches nothing
    grid = max(1, min(n_sm, total // NW))
    cs = Split(total, grid, 0)

    def cpu_of(li):
        return layers[li][0] + layers[li][1]

    def locate(c):
        li = 0
        while li + 1 < len(layers) and c >= begins[li + 1]:
            li += 1
        cpu = cpu_of(li)
        loc = c - begins[li]
        unit = loc // cpu
        return [li, unit, loc - unit * cpu, cpu]

    def step(r):
        r[2] += 1
        if r[2] < r[3]:
            return
        r[2] = 0
        r[1] += 1
        if r[1] < units:
            return
        r[1] = 0
        r[0] += 1
        while r[0] < len(layers) and cpu_of(r[0]) == 0:
            r[0] += 1
        r[3] = cpu_of(r[0]) if r[0] < len(layers) else 1

    holder = [None] * total
    finals = {}                       # (layer, unit) -> how it was written
    sdep = {}                         # (cta, warp, slot) -> (layer, unit)
    gdep = {}                         # (cta, slot) -> (layer, unit)
    scnt, gcnt = {}, {}               # tickets
    merges_s, merges_g = [], []       # (unit, slots read)

    for b in range(grid):
        C0, C1 = cs.first(b), cs.first(b + 1)
        assert C1 > C0, "every CTA holds a chunk (grid <= total / NW)"
        nvw = min(C1 - C0, NW)
        ws = Split(C1 - C0, nvw, C0)
        for warp in range(nvw):
            c0, c1 = ws.first(warp), ws.first(warp + 1)
            n = c1 - c0
            assert n >= 1
            cur = locate(c0)
            seg = -1
            for i in range(n):
                if i > 0:
                    step(cur)
                c = c0 + i
                assert cur == locate(c), "the stepped cursor equals a direct lookup"
                assert holder[c] is None
                holder[c] = (b, warp)
                if i == 0 or cur[2] == 0:
                    seg += 1
                if not (i == n - 1 or cur[2] == cur[3] - 1):
                    continue
                # finish(cur, seg)
                li, unit, _, cpu = cur
                key = (li, unit)
                ubeg = begins[li] + unit * cpu
                uend = ubeg + cpu
                if ubeg >= c0 and uend <= c1:
                    assert key not in finals
                    finals[key] = "warp"
                    continue
                lbeg, lend = max(ubeg, C0), min(uend, C1)
                cta_whole = ubeg >= C0 and uend <= C1
                wa, wb = ws.owner(lbeg), ws.owner(lend - 1)
                assert wa <= warp <= wb
                cslot = 0 if lbeg == C0 else 1
                to_global = True
                if wb > wa:
                    slot = (b, warp, 0 if seg == 0 else 1)
                    assert slot not in sdep, "a shared partial slot written twice"
                    sdep[slot] = key
                    t = scnt.get((b, wa), 0) + 1
                    scnt[(b, wa)] = t
                    if t != wb - wa + 1:
                        continue
                    wa_late = ws.first(wa) < lbeg
                    read = [(b, wa + k, 1 if (k == 0 and wa_late) else 0)
                            for k in range(wb - wa + 1)]
                    merges_s.append((key, read))
                    scnt[(b, wa)] = 0
                    if cta_whole:
                        assert key not in finals
                        finals[key] = "cta"
                        to_global = False
                assert to_global or cta_whole
                if not to_global:
                    continue
                assert not cta_whole, "a unit held by one CTA never goes to global memory"
                gslot = (b, cslot)
                assert gslot not in gdep, "a global partial slot written twice"
                gdep[gslot] = key
                ca, cb = cs.owner(ubeg), cs.owner(uend - 1)
                assert ca <= b <= cb
                t = gcnt.get(key, 0) + 1
                gcnt[key] = t
                if t != cb - ca + 1:
                    continue
                ca_late = cs.first(ca) < ubeg
                read = [(ca + k, 1 if (k == 0 and ca_late) else 0) for k in range(cb - ca + 1)]
                merges_g.append((key, read))
                assert key not in finals
                finals[key] = "grid"
                gcnt[key] = 0

    assert all(h is not None for h in holder), "every chunk processed"
    expected = {(li, u) for li in range(len(layers)) if cpu_of(li) > 0 for u in range(units)}
    assert set(finals) == expected, "every stored unit written exactly once"
    assert all(v == 0 for v in scnt.values()) and all(v == 0 for v in gcnt.values())
    for key, read in merges_s:
        assert [sdep.get(s) for s in read] == [key] * len(read), "shared merge reads its holders"
    for key, read in merges_g:
        assert [gdep.get(s) for s in read] == [key] * len(read), "global merge reads its CTAs"
    # the host's workspace check: two partial states per CTA
    assert max((s[0] for s in gdep), default=0) < grid
    return grid


def _random_layers(rng):
    layers = []
    for _ in range(rng.randint(1, 8)):
        bits = rng.choice([2, 4, 16])
        w = rng.randint(0, 9)
        p = 0 if bits == 16 else rng.choice([0, 0, 1, 2, 3, 16, 30, rng.randint(0, 60)])
        layers.append((w, p))
    return layers


def test_workload_shaped_layouts():
    """Chunk counts of the benchmark's workloads: long context (32 layers, 8 units,
    packed chunks 2..30 per unit, window chunks 5..8), the batched one (128 units,
    2 packed chunks, window 3..4), the quantize-only one (160 units, 1,024 packed
    chunks per unit at 4 bits; 4 of its layers)."""
    for NW in (8, 12):
        long_ctx = [(5 + l % 4, 30 - l * 28 // 31) for l in range(32)]
        assert replay(long_ctx, 8, NW, 152) == 152
        batched = [(3 + l % 2, 2) for l in range(32)]
        assert replay(batched, 128, NW, 152) == 152
        quant_only = [(1, 1024)] * 4          # 4 of its 40 layers
        assert replay(quant_only, 160, NW, 152) == 152


@pytest.mark.parametrize("seed", range(6))
def test_random_layouts(seed):
    rng = random.Random(seed)
    for _ in range(400):
        layers = _random_layers(rng)
        units = rng.choice([1, 2, 3, 4, 8, 16, 40, 64])
        replay(layers, units, rng.choice([8, 12]), rng.choice([1, 2, 3, 7, 19, 152]))


def test_degenerate_layouts():
    assert replay([(0, 0)], 4, 8, 152) == 0           # nothing stored
    assert replay([(1, 0)], 1, 8, 152) == 1           # one chunk: one CTA, one warp
    assert replay([(0, 0), (1, 0), (0, 0)], 1, 12, 152) == 1
    assert replay([(9, 0)], 1, 8, 152) == 1           # 9 chunks: one CTA of 8 warps
    assert replay([(0, 200)], 1, 8, 152) == 25        # one long unit over 25 CTAs
    assert replay([(0, 3)] * 64, 8192, 12, 152) == 152
