"""Pins for the oracle's E2-SCI path ("E2-SCI: Elastic Edge-Cloud Speculative
Decoding via Credit Inertia", paper notes, Key design 3): hand-computed
threshold and EWMA values (tests/golden/sci_recurrence.txt), the closed form
of the EWMA under a constant acceptance rate, and a brute-force window check
against scipy's Jensen-Shannon distance."""
import os

import numpy as np
import pytest
import scipy.special as sps
from scipy.spatial.distance import jensenshannon

import gen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    th, ew = [], []
    for line in open(os.path.join(GOLDEN, "sci_recurrence.txt")):
        if line.startswith("#") or not line.strip():
            continue
        kind, *v = line.split()
        (th if kind == "threshold" else ew).append(tuple(float(x) for x in v))
    return th, ew


@pytest.mark.parametrize("case", _golden()[0])
def test_threshold_golden(case):
    r, aw, T = case
    assert oracle.sci_threshold(r, oracle.SciParams(alpha_omega=aw)) == pytest.approx(T, abs=1e-15)


@pytest.mark.parametrize("case", _golden()[1])
def test_ewma_golden(case):
    r, p, r2 = case
    assert oracle.sci_ewma(r, p, 0.3) == pytest.approx(r2, abs=1e-15)


def test_ewma_constant_rate_closed_form():
    for c in (0.0, 0.25, 0.9, 1.0):
        r = 0.6
        for n in range(1, 30):
            r = oracle.sci_ewma(r, c, 0.3)
            assert r == pytest.approx(c + (0.6 - c) * 0.7 ** n, abs=1e-14)


def _straddling_window(rng, B, K, V, dtype):
    """Draft/target rows whose divergence spreads across the threshold range:
    target = draft + N(0, s^2) with s drawn per row from [0, 3]."""
    a = gen.store(rng.standard_normal((B, K + 1, V)) * 2.0, dtype)
    s = rng.uniform(0.0, 3.0, size=(B, K + 1, 1))
    t = gen.store(gen.widen(a, dtype).astype(np.float64) + s * rng.standard_normal((B, K + 1, V)), dtype)
    d = rng.integers(0, V, size=(B, K)).astype(np.int32)
    return a, t, d


@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_window_brute_force(dtype):
    rng = np.random.default_rng(14)
    B, K, V = 60, 4, 12
    a, t, d = _straddling_window(rng, B, K, V, dtype)
    r_hat = rng.uniform(0, 1, B)
    p = oracle.SciParams()
    res = oracle.sci_verify(a, t, d, r_hat, p)
    for r in range(B):
        T = min(max(0.3 + 0.2 * (r_hat[r] - 0.6), 0.1), 0.6)
        assert res.T[r] == pytest.approx(T, abs=1e-15)
        J = [jensenshannon(sps.softmax(gen.widen(a[r, i], dtype).astype(np.float64)),
                           sps.softmax(gen.widen(t[r, i], dtype).astype(np.float64))) ** 2
             for i in range(K + 1)]
        np.testing.assert_allclose(res.jsd[r], J, rtol=1e-9, atol=1e-14)
        n = next((i for i in range(K) if J[i] > T), K)
        assert res.accept_len[r] == n
        exp_tokens = list(d[r, :n]) + [int(np.argmax(gen.widen(t[r, n], dtype)))] + [-1] * (K - n)
        assert list(res.tokens[r]) == exp_tokens
        assert res.r_hat[r] == pytest.approx(0.7 * r_hat[r] + 0.3 * n / K, abs=1e-15)
    # the data exercises every outcome of the scan
    assert set(res.accept_len.tolist()) >= {0, 1, K}


def test_five_windows_state_carry_and_resume():
    """Five windows in a row equal two windows, a saved state, and three more."""
    B, K, V = 6, 8, 64
    wins = [gen.make_asymspec_batch("spiky", 100 + w, B, K, V, gen.BF16) for w in range(5)]
    r = np.full(B, 0.6)
    for w in wins:
        r = oracle.sci_verify(w.a, w.t, w.drafts, r).r_hat
    r2 = np.full(B, 0.6)
    for w in wins[:2]:
        r2 = oracle.sci_verify(w.a, w.t, w.drafts, r2).r_hat
    saved = r2.copy()
    r3 = saved
    for w in wins[2:]:
        r3 = oracle.sci_verify(w.a, w.t, w.drafts, r3).r_hat
    np.testing.assert_array_equal(r, r3)
