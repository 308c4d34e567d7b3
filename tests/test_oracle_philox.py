"""Pins for the oracle's Philox4x32-10: the published known-answer vectors
(tests/golden/philox4x32_10_kat.txt) and the uniformity of the derived floats."""
import os

import numpy as np
import pytest
from scipy import stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kat():
    rows = []
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        v = [int(x, 16) for x in line.split()]
        rows.append((v[0:4], v[4:6], v[6:10]))
    return rows


@pytest.mark.parametrize("case", _kat())
def test_philox_known_answers(case):
    ctr, key, out = case
    assert [int(x) for x in oracle.philox4x32_10(ctr, key)] == out


def test_uniform_from_word_range_and_fp32_exactness():
    for w in (0, 1, 511, 512, 0x7FFFFFFF, 0xFFFFFE00, 0xFFFFFFFF):
        u = oracle.uniform_from_word(w)
        assert 0.0 < u < 1.0
        assert float(np.float32(u)) == u
    assert oracle.uniform_from_word(0) == 2.0 ** -24
    assert oracle.uniform_from_word(0xFFFFFFFF) == 1.0 - 2.0 ** -24


def test_rapid_uniforms_are_uniform_and_distinct_per_stream():
    u = np.array([oracle.rapid_uniform(1234, 0, 1, r, i, k) for r in range(4) for i in range(5) for k in range(500)])
    assert stats.kstest(u, "uniform").pvalue > 1e-4
    # different streams / offsets / words give different numbers
    a = oracle.rapid_uniform(1234, 0, 0, 3, 2, 0)
    assert a != oracle.rapid_uniform(1234, 0, 1, 3, 2, 0)
    assert a != oracle.rapid_uniform(1234, 1, 0, 3, 2, 0)
    assert a != oracle.rapid_uniform(1234, 0, 0, 3, 2, 1)
    assert a != oracle.rapid_uniform(1235, 0, 0, 3, 2, 0)
