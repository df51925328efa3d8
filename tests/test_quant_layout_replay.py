"""A CPU replay of where the group quantizer writes each code, against where the
decode kernel and the exporter read it (index arithmetic only).

The quantizer (quant_device.cuh: `code_words`, `code_fragment`) loads a staged
16x16 tile with one 8x8-matrix load per tile (`ldmatrix .x4`; transposed for
values) and packs each lane's fragment elements into 32-bit words. Which element
a lane receives is fixed by the PTX ISA's fragment layout of `ldmatrix`: for the
plain form, lane l holds row l / 4 and columns 2 (l % 4), 2 (l % 4) + 1 of each
8x8 matrix; the transposed form delivers the same positions of the transposed
matrix. The readers use `kcode_pos` / `vcode_pos` (kvc_internal.cuh: the word
`(wi / 4) * 128 + 4 lane + wi % 4` and the bit `pair_bit(P) + 16 (odd)`), and the
parameters of each code come from the scratch slot `kq_pos` / `vq_pos`.

For every (token, channel) of a group, for head dims 64 and 128 and 2 and 4 bits,
this checks that the code is written to exactly the word and bit its readers
use, that no two elements share a field, and that it is quantized with the
scale and zero of its own group (key channel c; value token t and channels
32 gc ..)."""
import pytest

G = 32


# ---------------------------------------------------------------- readers
def pair_bit(P, bits):
    return 8 * (P // (8 // bits)) + bits * (P % (8 // bits))


def word_addr(lane, wi):
    return (wi >> 2) * 128 + lane * 4 + (wi & 3)


def kcode_pos(t, c, D, bits):
    mt, rl, gid = t >> 4, (t >> 3) & 1, t & 7
    ks, rh, tid, odd = c >> 4, (c >> 3) & 1, (c & 7) >> 1, c & 1
    KS = D >> 4
    if bits == 2:
        wi, P = mt * (KS >> 1) + (ks >> 1), 4 * rl + 2 * (ks & 1) + rh
    else:
        wi, P = mt * KS + ks, 2 * rl + rh
    return word_addr(gid * 4 + tid, wi), pair_bit(P, bits) + (16 if odd else 0)


def vcode_pos(t, c, D, bits):
    ks, rh, tid, odd = t >> 4, (t >> 3) & 1, (t & 7) >> 1, t & 1
    mt, rl, gid = c >> 4, (c >> 3) & 1, c & 7
    if bits == 2:
        wi, P = mt, 4 * rl + 2 * ks + rh
    else:
        wi, P = 2 * mt + ks, 2 * rl + rh
    return word_addr(gid * 4 + tid, wi), pair_bit(P, bits) + (16 if odd else 0)


def kq_pos(c):
    return ((c >> 4) * 4 + ((c & 7) >> 1)) * 4 + (c & 1) + 2 * ((c >> 3) & 1)


def vq_pos(t, gc):
    return ((gc * 2 + (t >> 4)) * 4 + ((t & 7) >> 1)) * 4 + (t & 1) + 2 * ((t >> 3) & 1)


# ---------------------------------------------------------------- writer
def ldmatrix_x4(rows0, cols0, lane, trans):
    """(row, col) in the staged tile of the two 16-bit elements that register k of
    `lane` receives, for the four 8x8 matrices whose top-left corners are
    (rows0[k], cols0[k]). Plain: row lane/4 of the matrix, columns 2 (lane%4) + e.
    Transposed: the same positions of the transposed matrix."""
    out = []
    for k in range(4):
        r, cc = lane >> 2, 2 * (lane & 3)
        if trans:
            out.append([(rows0[k] + cc + e, cols0[k] + r) for e in (0, 1)])
        else:
            out.append([(rows0[k] + r, cols0[k] + cc + e) for e in (0, 1)])
    return out


def writer(D, bits, kind):
    """{(token, channel): (word, bit, scratch slot)} as the quantizer writes them."""
    KS = D // 16
    TPW = D // 32
    TPWD = 1 if bits == 4 else 2
    WW = TPW // TPWD
    placed = {}
    for sub in range(4):                      # the four warps of the section
        wi0 = WW * sub
        for lane in range(32):
            tid = lane & 3
            for wj in range(WW):
                wi = wi0 + wj
                for s in range(TPWD):
                    if kind == 0:
                        if bits == 4:
                            mt, ks = wi // KS, wi % KS
                        else:
                            mt, ks = wi // (KS // 2), 2 * (wi % (KS // 2)) + s
                        # matrix m: tokens 16 mt (+8 for m = 2, 3), channels 16 ks (+8 for 1, 3)
                        rows0 = [16 * mt + 8 * (m >> 1) for m in range(4)]
                        cols0 = [16 * ks + 8 * (m & 1) for m in range(4)]
                        quad = ks * 4 + tid
                        frags = ldmatrix_x4(rows0, cols0, lane, trans=False)
                    else:
                        if bits == 4:
                            mt, ks = wi >> 1, wi & 1
                        else:
                            mt, ks = wi, s
                        # matrix m: tokens 16 ks (+8 for 1, 3), channels 16 mt (+8 for 2, 3)
                        rows0 = [16 * ks + 8 * (m & 1) for m in range(4)]
                        cols0 = [16 * mt + 8 * (m >> 1) for m in range(4)]
                        quad = ((mt >> 1) * 2 + ks) * 4 + tid
                        frags = ldmatrix_x4(rows0, cols0, lane, trans=True)
                    word = word_addr(lane, wi)
                    for k in range(4):
                        rh = k & 1
                        sh = 4 * k if bits == 4 else 8 * (k >> 1) + 2 * rh + 4 * s
                        for e, (tok, ch) in enumerate(frags[k]):
                            key = (tok, ch)
                            assert key not in placed, ("element written twice", key)
                            placed[key] = (word, sh + 16 * e, quad * 4 + 2 * rh + e)
    return placed


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bits", [2, 4])
def test_key_codes_land_where_they_are_read(D, bits):
    placed = writer(D, bits, 0)
    assert len(placed) == G * D
    fields = set()
    for (t, c), (word, bit, slot) in placed.items():
        assert 0 <= t < G and 0 <= c < D
        assert (word, bit) == kcode_pos(t, c, D, bits), (t, c)
        assert slot == kq_pos(c), "quantized with its own channel's parameters"
        assert 0 <= word < D * bits and bit + bits <= 32
        fields.add((word, bit))
    assert len(fields) == G * D


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bits", [2, 4])
def test_value_codes_land_where_they_are_read(D, bits):
    placed = writer(D, bits, 1)
    assert len(placed) == G * D
    fields = set()
    for (t, c), (word, bit, slot) in placed.items():
        assert 0 <= t < G and 0 <= c < D
        assert (word, bit) == vcode_pos(t, c, D, bits), (t, c)
        assert slot == vq_pos(t, c // 32), "quantized with its own group's parameters"
        assert 0 <= word < D * bits and bit + bits <= 32
        fields.add((word, bit))
    assert len(fields) == G * D


@pytest.mark.parametrize("D", [64, 128])
def test_scratch_slots_cover_each_group_once(D):
    """kq_pos is a permutation of the D key channels and vq_pos of the 32 x D/32
    value groups, inside the scratch's D slots per section."""
    assert sorted(kq_pos(c) for c in range(D)) == list(range(D))
    assert sorted(vq_pos(t, gc) for t in range(G) for gc in range(D // 32)) == list(range(D))
