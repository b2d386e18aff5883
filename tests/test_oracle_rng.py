"""Pins of the oracle's counter-based generator (Philox4x32-10) and uniforms."""
import numpy as np
import pytest
from scipy import stats

import oracle


def _kat(golden_dir):
    rows = []
    for line in open(f"{golden_dir}/philox4x32_10_kat.txt"):
        if line.strip() and not line.startswith("#"):
            rows.append([int(t, 16) for t in line.split()])
    return rows


def test_philox_known_answers(golden_dir):
    rows = _kat(golden_dir)
    assert len(rows) == 3
    for r in rows:
        out = oracle.philox4x32_10(r[0:4], r[4:6])
        assert [int(x) for x in out] == r[6:10]


def test_stream_layout_word_selection():
    # word col&3 of the call whose counter is (col>>2, row, step, domain)
    seed, step, dom, row = 0x0123456789ABCDEF, 5, 2, 77
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for col in (0, 1, 2, 3, 4, 9, 151935):
        out = oracle.philox4x32_10([col >> 2, row, step, dom], key)
        assert oracle.random_word(seed, step, dom, row, col) == int(out[col & 3])
    # the high half of step lands in counter word 3 above the domain bits
    out = oracle.philox4x32_10([0, 1, 7, 3 + 4 * 2], [9, 0])
    assert oracle.random_word(9, (2 << 32) + 7, 3, 1, 0) == int(out[0])


def test_uniform_exact_grid_and_range():
    for col in range(64):
        x = oracle.random_word(3, 0, 0, 0, col)
        u = oracle.uniform(3, 0, 0, 0, col)
        assert u == (2 * (x >> 9) + 1) / 2.0 ** 24
        assert 0.0 < u < 1.0
        assert float(np.float32(u)) == u           # exact in binary32
        g = oracle.gumbel(3, 0, 0, 0, col)
        assert g == pytest.approx(-np.log(-np.log(u)), abs=0, rel=1e-15)


def test_uniform_chi_square():
    n = 20000
    u = np.array([oracle.uniform(11, 1, 1, i, 0) for i in range(n)])
    counts, _ = np.histogram(u, bins=20, range=(0, 1))
    assert stats.chisquare(counts).pvalue > 1e-4
    # the Gumbel transform of the same stream has the standard Gumbel law
    g = -np.log(-np.log(u))
    assert stats.kstest(g, "gumbel_r").pvalue > 1e-4
