"""Pins of the exponent-code ablation (unary vs Huffman) and the stored
statistics of the synthetic workloads (tests/golden/exponent_stats.json,
written by tests/golden/make_exponent_stats.py from the oracle only)."""
import json
import os

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_huffman_lengths_kraft_and_bounds(orc):
    rng = np.random.default_rng(0)
    for _ in range(20):
        c = np.zeros(256)
        idx = rng.choice(256, rng.integers(2, 40), replace=False)
        c[idx] = rng.integers(1, 10000, idx.size)
        lens = orc.huffman_code_lengths(c)
        used = lens[c > 0]
        assert abs(np.sum(2.0 ** -used) - 1.0) < 1e-12          # full prefix code (Kraft equality)
        H = orc.exp_entropy(c)
        L = orc.huffman_mean_len(c)
        assert H - 1e-12 <= L < H + 1.0                          # Shannon: H <= L < H + 1
        _, roe = orc.rank_table(c)
        assert L <= orc.unary_mean_len(c, roe) + 1e-12            # Huffman is optimal among prefix codes


def test_huffman_dyadic_and_two_symbols(orc):
    c = np.zeros(256)
    c[[10, 11, 12, 13]] = [8, 4, 2, 2]                            # p = 1/2, 1/4, 1/8, 1/8
    assert list(orc.huffman_code_lengths(c)[[10, 11, 12, 13]]) == [1, 2, 3, 3]
    assert orc.huffman_mean_len(c) == pytest.approx(orc.exp_entropy(c))
    d = np.zeros(256)
    d[[0, 200]] = [5, 7]
    assert list(orc.huffman_code_lengths(d)[[0, 200]]) == [1, 1]
    # dyadic geometric p = 1/2, 1/4, ..., 1/256, 1/256: Huffman gives lengths
    # 1..8, 8 and unary 1..8, 9, so unary costs exactly the last symbol's
    # probability more
    g = np.zeros(256)
    g[100:108] = [2 ** (7 - i) for i in range(8)]
    g[108] = 1
    _, roe = orc.rank_table(g)
    assert list(orc.huffman_code_lengths(g)[100:109]) == [1, 2, 3, 4, 5, 6, 7, 8, 8]
    assert orc.unary_mean_len(g, roe) - orc.huffman_mean_len(g) == pytest.approx(1 / 256)


def test_stored_exponent_stats_match_oracle(orc):
    """The stored table is reproduced by the oracle (small workloads only)."""
    import synthetic
    stats = json.load(open(os.path.join(HERE, "golden", "exponent_stats.json")))
    w = synthetic.cfg0_weight().numpy().view(np.uint16)
    c = orc.exp_hist(w)
    _, roe = orc.rank_table(c)
    row = stats["cfg0_4096x4096_normal_outliers"]
    assert row["entropy_bits"] == pytest.approx(orc.exp_entropy(c), abs=1e-9)
    assert row["unary_mean_bits"] == pytest.approx(orc.unary_mean_len(c, roe), abs=1e-9)
    assert row["huffman_mean_bits"] == pytest.approx(orc.huffman_mean_len(c), abs=1e-9)
    for name, r in stats.items():
        assert r["entropy_bits"] <= r["huffman_mean_bits"] <= r["unary_mean_bits"] + 1e-12, name
