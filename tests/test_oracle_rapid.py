"""Pins for the oracle's RAPID path ("RAPID: Long-Context Inference with
Retrieval-Augmented Speculative Decoding", paper notes, Key designs 2-4):
the augmented logits equal one gradient step on T^2 KL(q || softmax(z/T))
(checked by finite differences, not by the printed gradient), eta = 0 reduces
to the target, tail/protection invariants, the exponential-race sampler's
distribution (chi-square), and the textbook result that with eta = 0 the
first emitted token is distributed as p when drafts are drawn from q."""
import math

import numpy as np
import pytest
import scipy.special as sps
from scipy import stats

import gen
import oracle


def _loss(z, q, T):
    p = sps.softmax(z / T)
    return T * T * float(np.sum(sps.rel_entr(q, p)))


@pytest.mark.parametrize("T", [1.0, 0.7, 2.0])
def test_zhat_is_one_gradient_step(T):
    rng = np.random.default_rng(11)
    V = 16
    z = (rng.standard_normal(V) * 2).astype(np.float32)
    # drafter probabilities with an exact sum of 1 (multiples of 1/64)
    w = np.append(rng.integers(1, 5, size=V - 1), 0).astype(np.float64)
    w[-1] = 64 - w.sum()
    assert w.sum() == 64 and np.all(w > 0)
    q = (w / 64).astype(np.float32)
    eta = 5.0
    row = oracle.rapid_row(z, q, T, eta)
    zd = z.astype(np.float64)
    h = 1e-5
    grad = np.array([(_loss(zd + h * np.eye(V)[k], q.astype(np.float64), T)
                      - _loss(zd - h * np.eye(V)[k], q.astype(np.float64), T)) / (2 * h) for k in range(V)])
    np.testing.assert_allclose(row.zhat - zd, -eta * grad, atol=2e-8)


def test_eta_zero_and_invariants():
    rng = np.random.default_rng(12)
    b = gen.make_rapid_batch(5, 2, 2, 3000)
    for eta in (0.0, 5.0, 20.0, 50.0):
        for r in range(2):
            for i in range(3):
                z, q = b.z[r, i], b.q[r, i]
                row = oracle.rapid_row(z, q, 1.0, eta, 0.1)
                np.testing.assert_allclose(row.p, sps.softmax(z.astype(np.float64)), rtol=1e-12, atol=1e-300)
                if eta == 0.0:
                    np.testing.assert_allclose(row.phat, row.p, rtol=1e-12, atol=1e-300)
                    np.testing.assert_allclose(row.prot, row.p, rtol=1e-12, atol=1e-300)
                thr = 0.1 * row.phat.max()
                tail = row.phat < thr
                assert row.ntail == int(tail.sum())
                assert np.all(row.prot[tail] == row.p[tail])             # tail keeps p exactly
                assert math.isclose(row.prot.sum(), 1.0, rel_tol=0, abs_tol=1e-12)
                head = ~tail
                ratio = row.prot[head] / row.phat[head]
                np.testing.assert_allclose(ratio, ratio[0], rtol=1e-12)   # head rescaled uniformly
                assert head[np.argmax(row.phat)]


def test_residual_reduces_to_textbook_at_eta_zero():
    b = gen.make_rapid_batch(6, 1, 1, 500)
    row = oracle.rapid_row(b.z[0, 0], b.q[0, 0], 1.0, 0.0)
    q = b.q[0, 0].astype(np.float64)
    r = np.maximum(np.maximum(row.p - row.prot, row.p - q), 0)
    np.testing.assert_allclose(r, np.maximum(row.p - q, 0), atol=1e-15)
    assert r.sum() > 0 and math.isclose((r / r.sum()).sum(), 1.0)


def test_race_distribution_chi_square():
    w = np.array([0.05, 0.0, 0.3, 0.15, 0.0, 0.2, 0.25, 0.05])
    counts = np.zeros(len(w))
    n = 0
    for req in range(200):
        for row in range(100):
            k, _ = oracle.race(w, 1234, 0, 1, req, row)
            counts[k] += 1
            n += 1
    assert counts[1] == 0 and counts[4] == 0                  # zero weight never wins
    nz = w > 0
    p = stats.chisquare(counts[nz], n * w[nz] / w.sum()).pvalue
    assert p > 1e-4
    k, _ = oracle.race(np.zeros(5), 1, 0, 1, 0, 0)
    assert k == -1


def test_eta_zero_first_token_marginal_is_target():
    """Standard speculative sampling: draft d ~ q, accept with u*q(d) < p(d), else draw
    from norm(max(p - q, 0)).  The first emitted token is then distributed as p."""
    rng = np.random.default_rng(13)
    V, B = 12, 20000
    z = (rng.standard_normal(V) * 1.5).astype(np.float32)
    q = sps.softmax(z.astype(np.float64) + rng.standard_normal(V)).astype(np.float32)
    qd = q.astype(np.float64) / q.astype(np.float64).sum()
    zz = np.broadcast_to(z, (B, 2, V)).copy()
    qq = np.broadcast_to(q, (B, 2, V)).copy()
    d = rng.choice(V, size=(B, 1), p=qd).astype(np.int32)
    res = oracle.rapid_verify(zz, qq, d, 1.0, 0.0, 0.1, 777)
    first = res.tokens[:, 0]
    p = sps.softmax(z.astype(np.float64))
    counts = np.bincount(first, minlength=V)
    assert stats.chisquare(counts, B * p).pvalue > 1e-4
    assert 0 < res.accept_len.mean() < 1


def test_verify_scan_structure():
    b = gen.make_rapid_batch(1234, 4, 10, 2000)
    for eta in (0.0, 10.0):
        res = oracle.rapid_verify(b.z, b.q, b.drafts, 1.0, eta, 0.1, 1234)
        for r in range(4):
            n = res.accept_len[r]
            assert 0 <= n <= 10
            assert list(res.tokens[r, :n]) == list(b.drafts[r, :n])
            assert 0 <= res.tokens[r, n] < 2000
            assert np.all(res.tokens[r, n + 1:] == -1)
            # the accept test, restated from the row quantities
            for i in range(n + (1 if n < 10 else 0)):
                row = oracle.rapid_row(b.z[r, i], b.q[r, i], 1.0, eta, 0.1)
                u = oracle.rapid_uniform(1234, 0, 0, r, i, 0)
                dd = b.drafts[r, i]
                assert (u * float(b.q[r, i, dd]) < row.prot[dd]) == (i < n)


# ------------------------------------------------------------------ the other tail-protection reading

def _tail_case(seed, V=200, eta=10.0):
    rng = np.random.default_rng(seed)
    z = (2.0 * rng.standard_normal(V) - 1.1 * np.log(rng.permutation(V) + 1.0)).astype(np.float32)
    q = sps.softmax(z.astype(np.float64) + rng.standard_normal(V)).astype(np.float32)
    return z, q, eta


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_renormalised_tail_reading(seed):
    """tail_mode 1: p substitutes phat on the tail, then every entry is renormalised, so the
    protected target is w / sum(w) with w = p on the tail and phat on the head."""
    z, q, eta = _tail_case(seed)
    r0 = oracle.rapid_row(z, q, 1.0, eta, 0.1, tail_mode=0)
    r1 = oracle.rapid_row(z, q, 1.0, eta, 0.1, tail_mode=1)
    np.testing.assert_array_equal(r0.p, r1.p)
    np.testing.assert_array_equal(r0.phat, r1.phat)
    tail = r1.phat < 0.1 * r1.phat.max()
    assert 0 < tail.sum() < len(z)
    assert r1.prot.sum() == pytest.approx(1.0, abs=1e-12)
    # one common factor 1/Z on both sides of the boundary
    ratios = np.concatenate([r1.prot[tail] / r1.p[tail], r1.prot[~tail] / r1.phat[~tail]])
    np.testing.assert_allclose(ratios, ratios[0], rtol=1e-12)
    # unlike the default reading, the tail is scaled too (Z != 1 here)
    assert abs(ratios[0] - 1.0) > 1e-6
    np.testing.assert_allclose(r0.prot[tail], r0.p[tail], rtol=0, atol=0)


def test_renormalised_tail_reading_eta_zero_is_p():
    z, q, _ = _tail_case(7)
    r1 = oracle.rapid_row(z, q, 1.0, 0.0, 0.1, tail_mode=1)
    np.testing.assert_allclose(r1.prot, r1.p, rtol=1e-12, atol=0)
