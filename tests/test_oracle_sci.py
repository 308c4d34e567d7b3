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


# ------------------------------------------------------------------ stabilisers

def _stab_golden():
    rows = []
    with open(os.path.join(GOLDEN, "sci_stabilisers.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                w, n, T, r = line.split()
                rows.append((int(w), int(n), float(T), float(r)))
    return rows


def _scripted_window(rng, n, K, V):
    """Rows before n: draft == target (J = 0, accepted at any T >= 0); row n (if n < K): disjoint
    spikes (J close to ln 2, rejected at any T <= 0.6)."""
    draft = rng.standard_normal((1, K + 1, V)).astype(np.float32)
    target = draft.copy()
    if n < K:
        draft[0, n, :] = -50.0
        target[0, n, :] = -50.0
        draft[0, n, 0] = 50.0
        target[0, n, 1] = 50.0
    return draft, target, np.zeros((1, K), np.int32)


def test_stabiliser_golden_sequence():
    rng = np.random.default_rng(5)
    stab = oracle.SciStabilisers(hysteresis=0.02, min_refresh=2, fallback_acc=0.3, fallback_T=0.12)
    state = oracle.sci_state(1)
    r_hat = np.array([0.6])
    for w, n, T_exp, r_exp in _stab_golden():
        draft, target, d = _scripted_window(rng, n, 4, 16)
        out = oracle.sci_verify(draft, target, d, r_hat, stab=stab, state=state)
        assert out.accept_len[0] == n, w
        assert out.T[0] == pytest.approx(T_exp, abs=1e-12), w
        assert out.r_hat[0] == pytest.approx(r_exp, abs=1e-12), w
        r_hat = out.r_hat


def test_stabiliser_rule_cases():
    s = oracle.SciStabilisers(hysteresis=0.05, min_refresh=3, fallback_acc=0.5, fallback_T=0.11)
    st = oracle.sci_state(1)[0]
    assert oracle.sci_stab_threshold(st, 0.33, s) == (0.33, 1)          # first window takes the candidate
    st.flags, st.T_applied, st.age = 1, 0.30, 2
    assert oracle.sci_stab_threshold(st, 0.40, s) == (0.30, 3)          # refresh interval not reached
    st.age = 3
    assert oracle.sci_stab_threshold(st, 0.34, s) == (0.30, 4)          # inside the hysteresis band
    assert oracle.sci_stab_threshold(st, 0.36, s) == (0.36, 1)          # outside it: change
    assert oracle.sci_stab_threshold(st, 0.24, s) == (0.24, 1)          # the band works both ways
    st.flags = 3
    assert oracle.sci_stab_threshold(st, 0.50, s) == (0.11, 1)          # fallback pending wins


def test_stabilisers_off_equal_plain_windows():
    rng = np.random.default_rng(8)
    B, K, V = 6, 4, 300
    off = oracle.SciStabilisers(hysteresis=0.0, min_refresh=1, fallback_acc=0.0, fallback_T=0.1)
    state = oracle.sci_state(B)
    r_a = np.full(B, 0.6)
    r_b = r_a.copy()
    for w in range(4):
        draft, target, d = _straddling_window(rng, B, K, V, gen.F32)
        a = oracle.sci_verify(draft, target, d, r_a)
        b = oracle.sci_verify(draft, target, d, r_b, stab=off, state=state)
        np.testing.assert_array_equal(a.accept_len, b.accept_len)
        np.testing.assert_array_equal(a.tokens, b.tokens)
        np.testing.assert_array_equal(a.T, b.T)
        np.testing.assert_array_equal(a.r_hat, b.r_hat)
        r_a, r_b = a.r_hat, b.r_hat
