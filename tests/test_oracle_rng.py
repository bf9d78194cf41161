"""Pins for the oracle's random stream: Philox4x32-10 and the two variates derived from it.

The Philox bijection is pinned to the known-answer vectors published with Salmon et al.
(SC'11). The accept uniform u and the race variate E are pinned to their distributions:
u uniform on the 2^-24 grid of [0, 1) and E exponential with mean 1, which a wrong shift,
scale, sign or log base would break.
"""

import math

import numpy as np
import pytest
from scipy import stats

import oracle
from conftest import read_table
from pyref import e_race, philox, u_accept


def test_philox_known_answers():
    rows = read_table("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for row in rows:
        vals = [int(v, 16) for v in row]
        ctr, key, want = vals[0:4], vals[4:6], vals[6:10]
        got = oracle.philox4x32_10(ctr, key)
        assert [int(v) for v in got] == want
        # the independent pure-Python statement agrees too
        assert philox(ctr, key) == want


def test_accept_uniform_distribution():
    us = np.array([oracle.accept_uniform(12345, r, j) for r in range(4000) for j in range(8)])
    # on the 2^-24 grid, inside [0, 1)
    assert np.all(us >= 0.0) and np.all(us < 1.0)
    assert np.all(np.floor(us * 2**24) == us * 2**24)
    ks = stats.kstest(us, "uniform")
    assert ks.pvalue > 1e-3
    assert abs(us.mean() - 0.5) < 4 * math.sqrt(1 / 12 / us.size)


def test_race_variate_is_exponential():
    es = np.array([oracle.race_E(777, r, j, x) for r in range(50) for j in range(4)
                   for x in range(1000)], dtype=np.float64)
    assert np.all(es > 0.0)
    # the smallest and largest attainable values: v in [2^-33, 1 - 2^-33]
    assert es.max() <= -math.log(2.0**-33) * (1 + 1e-6)
    ks = stats.kstest(es, "expon")
    assert ks.pvalue > 1e-3
    assert abs(es.mean() - 1.0) < 4 / math.sqrt(es.size)


def test_race_variate_counter_layout():
    # four consecutive vocab entries share one Philox block (words 0..3 of block x >> 2, tag 1)
    seed, r, j = 0xDEADBEEF12345678, 7, 3
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for x0 in (0, 4, 1024, 201084):
        words = philox([x0 >> 2, j, r, 1], key)
        for t in range(4):
            w = words[t]
            want = np.float32(-math.log((w + 0.5) / 2**32))
            assert oracle.race_E(seed, r, j, x0 + t) == want
            assert e_race(seed, r, j, x0 + t) == want
    # accept uniform: word 0 of block (0, j, r, 0)
    w = philox([0, j, r, 0], key)[0]
    assert oracle.accept_uniform(seed, r, j) == (w >> 8) / 2**24 == u_accept(seed, r, j)


@pytest.mark.parametrize("seed", [0, 1, 2**40 + 5])
def test_streams_differ_by_request_row_and_seed(seed):
    a = [oracle.race_E(seed, 0, 0, x) for x in range(64)]
    b = [oracle.race_E(seed, 1, 0, x) for x in range(64)]
    c = [oracle.race_E(seed, 0, 1, x) for x in range(64)]
    d = [oracle.race_E(seed + 1, 0, 0, x) for x in range(64)]
    assert a != b and a != c and a != d
