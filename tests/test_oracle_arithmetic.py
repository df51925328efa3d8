"""Pins the oracle's cache-size arithmetic to the numbers the pages print."""
import os
from fractions import Fraction

from oracle import blog_budget_row, minikv_sizes


def _rows(path):
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split("|")


def test_blog_budget_table(golden_dir):
    """Every row of the blog's worked Llama-2-13B budget table, exactly."""
    L, D, CTX = 40, 128, 32_768
    baseline = blog_budget_row(L, 40, D, 16)
    rows = list(_rows(os.path.join(golden_dir, "blog_budget_llama2_13b.txt")))
    assert len(rows) == 6
    for label, bits, frac, heads, bpt, gib, rel in rows:
        bits, heads = int(bits), int(heads)
        quantized = bits < 16
        stored = bits - 1 if quantized else bits        # the table folds scales into bits
        b = blog_budget_row(L, heads, D, stored, Fraction(frac), quantized=quantized)
        assert b == int(bpt.replace(",", "")), label
        assert f"{float(b * CTX / 2**30):.2f}" == gib, label
        assert f"{float(b / baseline):.1%}" == rel, label


def test_llama2_13b_headline_numbers():
    """819,200 B/token BF16, 153,600 B/token 2-bit+scales, 25.00 GiB per 32k sequence."""
    assert blog_budget_row(40, 40, 128, 16) == 819_200
    assert blog_budget_row(40, 40, 128, 2, quantized=True) == 153_600
    assert blog_budget_row(40, 40, 128, 4, quantized=True) == 256_000
    assert blog_budget_row(40, 40, 128, 16) * 32_768 == 25 * 2**30


def test_minikv_worked_example(golden_dir):
    """MiniKV §5.2: 2.4 GB full vs 0.33 GB MiniKV (86%), H2O at 15% = 0.32 GB."""
    s = minikv_sizes(32, 4096, 4096, 512)
    assert s["full"] == 2_415_919_104
    assert s["minikv"] == 335_544_320
    assert int(s["h2o"]) == 322_122_547
    printed = {r[0]: r[1] for r in _rows(os.path.join(golden_dir, "minikv_sizes.txt"))}

    def shown(value, text):
        """The page prints values cut (not rounded) to the digits it shows."""
        step = 10.0 ** -len(text.split(".")[1]) if "." in text else 1.0
        return float(text) <= value < float(text) + step

    assert shown(float(s["full"]) / 1e9, printed["full"])
    assert shown(float(s["minikv"]) / 1e9, printed["minikv"])
    assert shown(float(s["h2o"]) / 1e9, printed["h2o"])
    assert shown(100 * (1 - float(s["minikv"] / s["full"])), printed["compression"])
    # KIVI at group 16: 4 bytes of codes + 4 bytes of fp16 scale/zero per 16 numbers
    assert s["kivi"] == 32 * 4096 * (4096 + 512)


def test_two_bit_group32_counts_one_extra_bit():
    """A 16-bit scale + 16-bit zero per 32 numbers is exactly one bit per number."""
    assert blog_budget_row(1, 1, 32, 2, quantized=True) == blog_budget_row(1, 1, 32, 3)
