"""Pins for the CPU oracle's AsymSpec path, each against something other than the
oracle itself: library routines (scipy logsumexp / softmax / entropy /
jensenshannon, numpy argmax), closed forms derived by hand (tests/golden),
the bounds and reductions stated in "AsymSpec: Context-Asymmetric Speculative
Decoding for Agentic LLMs" (reading notes) sec. 4.1-4.2, and brute force over
every draft id at small V in the probability domain."""
import math
import os

import numpy as np
import pytest
import scipy.special as sps
from scipy.spatial.distance import jensenshannon
from scipy.stats import entropy

import gen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(rng, n, V, dtype, scale=2.0):
    x = rng.standard_normal((n, V)) * scale
    return gen.store(x, dtype)


def _w(x, dtype):
    return gen.widen(x, dtype).astype(np.float64)


@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_lse_matches_scipy(dtype):
    rng = np.random.default_rng(1)
    for V in (1, 2, 7, 16, 1000, 32000):
        x = _rows(rng, 1, V, dtype, 3.0)[0]
        assert oracle.lse(x) == pytest.approx(sps.logsumexp(_w(x, dtype)), rel=1e-13, abs=1e-13)


def test_lse_special_cases():
    x = np.array([-np.inf, -np.inf], np.float32)
    assert oracle.lse(x) == -np.inf
    assert oracle.lse(np.array([3.25], np.float32)) == 3.25
    # shift invariance with exactly representable shifts
    rng = np.random.default_rng(2)
    x = np.round(rng.standard_normal(257) * 64) / 64
    x32 = x.astype(np.float32)
    assert oracle.lse(x32 + np.float32(5.0)) == pytest.approx(oracle.lse(x32) + 5.0, abs=1e-12)
    # temperature scale: lse(x / T)
    assert oracle.lse(x32, 0.5) == pytest.approx(sps.logsumexp(x32.astype(np.float64) / 2.0), abs=1e-12)


def _golden_jsd():
    out = []
    for line in open(os.path.join(GOLDEN, "jsd_closed_forms.txt")):
        if line.startswith("#") or not line.strip():
            continue
        name, a, b, v = [s.strip() for s in line.split("|")]
        out.append((name, np.array([float(s) for s in a.split()], np.float32),
                    np.array([float(s) for s in b.split()], np.float32), float(v)))
    return out


@pytest.mark.parametrize("case", _golden_jsd(), ids=lambda c: c[0])
def test_jsd_closed_forms(case):
    _, a, b, v = case
    assert oracle.jsd(a, b) == pytest.approx(v, abs=1e-15)


@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_jsd_matches_library(dtype):
    rng = np.random.default_rng(3)
    for V in (2, 3, 16, 257, 5000):
        a = _rows(rng, 1, V, dtype)[0]
        b = _rows(rng, 1, V, dtype)[0]
        p = sps.softmax(_w(a, dtype))
        q = sps.softmax(_w(b, dtype))
        ref = jensenshannon(p, q) ** 2            # natural log by default
        ref2 = entropy(0.5 * (p + q)) - 0.5 * (entropy(p) + entropy(q))
        D = oracle.jsd(a, b)
        assert D == pytest.approx(ref, rel=1e-9, abs=1e-14)
        assert D == pytest.approx(ref2, rel=1e-9, abs=1e-14)


def test_jsd_bounds_identity_and_disjoint():
    rng = np.random.default_rng(4)
    for _ in range(50):
        V = int(rng.integers(2, 64))
        a = _rows(rng, 1, V, gen.F32, float(rng.uniform(0.1, 20)))[0]
        b = _rows(rng, 1, V, gen.F32, float(rng.uniform(0.1, 20)))[0]
        D = oracle.jsd(a, b)
        assert -1e-15 <= D <= math.log(2) + 1e-15
        assert oracle.jsd(a, a) == 0.0                       # a == b gives exactly 0
    # one-hot spikes far apart approach ln 2
    a = np.zeros(32, np.float32); a[3] = 60
    b = np.zeros(32, np.float32); b[17] = 60
    assert abs(oracle.jsd(a, b) - math.log(2)) < 1e-12
    # symmetry
    x, y = _rows(rng, 2, 100, gen.BF16)
    assert oracle.jsd(x, y) == pytest.approx(oracle.jsd(y, x), rel=1e-14)


def _exact_score(a, b, t, beta, dtype, src=0):
    """t + beta * delta in float64 from the exactly widened stored values (the definition)."""
    af, bf, tf = (gen.widen(x, dtype).astype(np.float64) for x in (a, b, t))
    d = {0: af - bf, 1: af, 2: tf - bf}[src]
    return tf + np.float64(np.float32(beta)) * d


@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_fused_argmax_matches_numpy(dtype):
    rng = np.random.default_rng(5)
    for beta in (0.0, 1.0, 1.5, -0.75):
        for V in (1, 2, 9, 16, 4097):
            a, b, t = _rows(rng, 3, V, dtype)
            assert oracle.fused_argmax(a, b, t, beta) == int(np.argmax(_exact_score(a, b, t, beta, dtype)))


def test_fused_argmax_is_shift_invariant_and_ignores_equal_drafters():
    """Adding a constant to t (exactly representable) or to both a and b leaves the winner; with
    a == b the score is t itself (ASYM sec. 4.1: no context gain, no steering)."""
    rng = np.random.default_rng(15)
    for _ in range(20):
        a, b, t = _rows(rng, 3, 777, gen.F32)
        k = oracle.fused_argmax(a, b, t, 1.5)
        assert oracle.fused_argmax(a, b, t + np.float32(8.0), 1.5) == k or oracle.fused_argmax_near(a, b, t, 1.5)[1]
        assert oracle.fused_argmax(a, a, t, 2.0) == int(np.argmax(t))


def test_fused_argmax_near_tie_under_single_precision():
    """A row built so that the exact scores differ by 2^-30 while the single-precision evaluation
    rounds both to the same value: the exact argmax is entry 1, the fp32 evaluation picks entry 0
    (lowest index of equal values), and the oracle flags the row as a near tie."""
    a = np.array([1 + 2 ** -23, 1 + 2 ** -23, -3.0], np.float32)
    b = np.array([2 ** -30, 0.0, 0.0], np.float32)
    t = np.zeros(3, np.float32)
    assert float(a[0]) - float(b[0]) < float(a[1]) - float(b[1])          # exact order: entry 1 wins
    assert np.float32(a[0] - b[0]) == np.float32(a[1] - b[1])             # fp32 difference: a tie
    k, near = oracle.fused_argmax_near(a, b, t, 1.0)
    assert (k, near) == (1, True)
    assert oracle.fused_argmax_fp32(a, b, t, 1.0) == 0
    # the same rows spread apart by more than the rounding bound: no flag
    b2 = np.array([2 ** -10, 0.0, 0.0], np.float32)
    assert oracle.fused_argmax_near(a, b2, t, 1.0) == (1, False)
    # an exact tie of single-precision scores is decided by the index rule and not flagged
    t3 = np.array([2.0, 2.0, 0.5], np.float32)
    z = np.zeros(3, np.float32)
    assert oracle.fused_argmax_near(z, z, t3, 1.0) == (0, False)
    # an exact tie whose delta is not a single-precision number is flagged (rounding could reorder it)
    a4 = np.array([1.0, 1.0 + 2 ** -23], np.float32)
    b4 = np.array([2 ** -40, 2 ** -23 + 2 ** -40], np.float32)
    t4 = np.zeros(2, np.float32)
    s4 = _exact_score(a4, b4, t4, 1.0, gen.F32)
    assert s4[0] == s4[1]
    assert oracle.fused_argmax_near(a4, b4, t4, 1.0) == (0, True)


@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_single_precision_winners_differ_only_on_near_ties(dtype):
    """Over many random rows (values spread so that near ties happen), every row where the
    single-precision evaluation picks another entry than the exact argmax is flagged near."""
    rng = np.random.default_rng(16 + dtype)
    differ = 0
    for _ in range(300):
        V = int(rng.integers(2, 40))
        a = gen.store(np.round(rng.standard_normal(V) * 8) / 8 + rng.standard_normal(V) * 1e-6, dtype)
        b = gen.store(np.round(rng.standard_normal(V) * 8) / 8, dtype)
        t = gen.store(np.round(rng.standard_normal(V) * 8) / 8, dtype)
        beta = float(rng.choice([1.0, 1.5, 2.0, 0.3]))
        k, near = oracle.fused_argmax_near(a, b, t, beta)
        if oracle.fused_argmax_fp32(a, b, t, beta) != k:
            differ += 1
            assert near
    # fp32 inputs: the 1e-6 perturbations survive storage and some rows do differ; bf16 storage
    # rounds them away (every score is then a single-precision number and the two always agree)
    assert differ >= 1 if dtype == gen.F32 else differ == 0


def test_fused_argmax_ties_and_nan():
    t = np.array([1, 5, 5, 2, 5], np.float32)
    z = np.zeros(5, np.float32)
    assert oracle.fused_argmax(z, z, t, 1.0) == 1                  # lowest index among ties
    t2 = np.array([np.nan, 1, 3, np.nan, 3], np.float32)
    assert oracle.fused_argmax(z, z, t2, 0.0) == 2                 # NaN never wins
    ninf = np.full(4, -np.inf, np.float32)
    assert oracle.fused_argmax(z[:4], z[:4], ninf, 0.0) == 0       # no finite score: index 0
    t3 = np.array([-np.inf, -np.inf, -2.0, -np.inf], np.float32)
    assert oracle.fused_argmax(z[:4], z[:4], t3, 0.0) == 2
    # beta = 0 reduces to argmax t
    rng = np.random.default_rng(6)
    a, b, t = _rows(rng, 3, 1000, gen.BF16)
    assert oracle.fused_argmax(a, b, t, 0.0) == int(np.argmax(gen.widen(t, gen.BF16)))


# ------------------------------------------------------------------ brute force

def _brute_request(a, b, t, drafts, beta, gamma, dtype):
    """Probability-domain restatement: accept iff p_t[d] > gamma * exp(-D) * p_b[d].
    beta and gamma cross the boundary as fp32, so they are rounded the same way here."""
    gamma = float(np.float32(gamma))
    K = len(drafts)
    n = K
    margins = []
    for i in range(K):
        aw, bw, tw = _w(a[i], dtype), _w(b[i], dtype), _w(t[i], dtype)
        pa, pb, pt = sps.softmax(aw), sps.softmax(bw), sps.softmax(tw)
        D = jensenshannon(pa, pb) ** 2
        lhs, rhs = pt[drafts[i]], gamma * math.exp(-D) * pb[drafts[i]]
        margins.append(math.log(lhs) - math.log(rhs) if lhs > 0 and rhs > 0 else np.inf)
        if not lhs > rhs:
            n = i
            break
    s = _exact_score(a[n], b[n], t[n], beta, dtype)
    tokens = [int(x) for x in drafts[:n]] + [int(np.argmax(s))] + [-1] * (K - n)
    return n, tokens, margins


@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_verify_brute_force_every_draft(dtype):
    """Every draft id d in [0, V) at the first position, V <= 16, several (beta, gamma)."""
    rng = np.random.default_rng(7)
    checked = flagged = 0
    for trial in range(12):
        V = int(rng.integers(2, 17))
        K = int(rng.integers(1, 4))
        a = _rows(rng, K + 1, V, dtype, 1.5)
        b = gen.store(_w(a, dtype) + rng.standard_normal(a.shape) * rng.uniform(0, 1.5), dtype)
        t = gen.store(_w(b, dtype) + rng.standard_normal(a.shape), dtype)
        beta, gamma = [(1.0, 0.5), (0.0, 1.0), (2.0, 0.4), (1.5, 0.7)][trial % 4]
        for d0 in range(V):
            drafts = rng.integers(0, V, size=K).astype(np.int32)
            drafts[0] = d0
            res = oracle.asymspec_verify(a[None], b[None], t[None], drafts[None], beta, gamma)
            n, tokens, margins = _brute_request(a, b, t, drafts, beta, gamma, dtype)
            if res.flags[0] & (oracle.FLAG_NEAR_MARGIN | oracle.FLAG_NEAR_TIE):
                flagged += 1
                continue
            checked += 1
            assert res.accept_len[0] == n
            assert list(res.tokens[0]) == tokens
            for i, m in enumerate(margins):
                if np.isfinite(m):
                    assert res.margin[0, i] == pytest.approx(m, abs=1e-9)
    assert checked > 100 and flagged < checked / 10


def test_gamma_eff_bounds_and_degenerate_run():
    """gamma_eff = gamma * exp(-D) lies in [gamma/2, gamma]; with beta = 0 the emitted
    token is argmax t; with a == b, D = 0 and the gate is p_t(d) > gamma * p_b(d)."""
    rng = np.random.default_rng(8)
    batch = gen.make_asymspec_batch("spiky", 99, 24, 3, 600, gen.F32, identical_frac=0.3)
    for beta, gamma in [(1.0, 0.5), (0.0, 1.0)]:
        res = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, beta, gamma)
        geff = gamma * np.exp(-res.D)
        assert np.all(geff >= gamma / 2 - 1e-15) and np.all(geff <= gamma + 1e-15)
        for r in range(batch.B):
            n = res.accept_len[r]
            tok = res.tokens[r, n]
            if beta == 0.0 or batch.identical[r]:
                assert tok == int(np.argmax(gen.widen(batch.t[r, n], gen.F32)))
            if batch.identical[r]:
                assert np.all(res.D[r] == 0.0)
                for i in range(n + (1 if n < 3 else 0)):
                    if i >= 3:
                        break
                    d = batch.drafts[r, i]
                    lt = res.lse[r, i, 2]; lb = res.lse[r, i, 1]
                    pt = math.exp(float(gen.widen(batch.t[r, i], gen.F32)[d]) - lt)
                    pb = math.exp(float(gen.widen(batch.b[r, i], gen.F32)[d]) - lb)
                    assert (pt > gamma * pb) == (i < n)
    # the accept lengths differ between the two runs on at least one request
    r1 = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.0, 0.5)
    r0 = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 0.0, 1.0)
    assert np.any(r1.accept_len != r0.accept_len) or np.any(r1.tokens != r0.tokens)


def test_flags_nonfinite_and_bad_draft():
    rng = np.random.default_rng(9)
    a, b, t = (_rows(rng, 3, 20, gen.F32).reshape(1, 3, 20) for _ in range(3))
    d = np.array([[1, 2]], np.int32)
    a2 = a.copy(); a2[0, 1, 5] = np.nan
    r = oracle.asymspec_verify(a2, b, t, d, 1.0, 0.5)
    assert r.flags[0] & oracle.FLAG_NONFINITE and r.accept_len[0] == 0 and np.all(r.tokens == -1)
    t2 = t.copy(); t2[0, 2, 0] = np.inf
    assert oracle.asymspec_verify(a, b, t2, d, 1.0, 0.5).flags[0] & oracle.FLAG_NONFINITE
    b2 = b.copy(); b2[0, 0, 3] = -np.inf                      # -inf is a legal logit
    assert not oracle.asymspec_verify(a, b2, t, d, 1.0, 0.5).flags[0] & oracle.FLAG_NONFINITE
    b3 = b.copy(); b3[0, 1, :] = -np.inf                      # ... but a row of -inf has no softmax
    assert oracle.asymspec_verify(a, b3, t, d, 1.0, 0.5).flags[0] & oracle.FLAG_NONFINITE
    r = oracle.asymspec_verify(a, b, t, np.array([[1, 20]], np.int32), 1.0, 0.5)
    assert r.flags[0] & oracle.FLAG_BAD_DRAFT and np.all(r.tokens == -1)


def test_gate_is_strict():
    """With t == b and gamma = 1 both sides of the printed inequality are equal
    (D = 0 when a == b), so the strict test rejects the first draft."""
    rng = np.random.default_rng(10)
    a = _rows(rng, 3, 50, gen.BF16).reshape(1, 3, 50)
    d = np.array([[4, 9]], np.int32)
    r = oracle.asymspec_verify(a, a, a, d, 1.0, 1.0)
    assert r.margin[0, 0] == 0.0 and r.accept_len[0] == 0
    assert r.flags[0] & oracle.FLAG_NEAR_MARGIN


@pytest.mark.parametrize("src", [0, 1, 2])
def test_delta_source_ablation_argmax(src):
    """ASYM sec. 5 ablation: delta := a - b (method), a (raw), t - b (two-model difference);
    checked against numpy argmax of the exact score."""
    rng = np.random.default_rng(30 + src)
    for dtype in (gen.F32, gen.BF16):
        for beta in (0.0, 1.0, 2.0):
            a, b, t = _rows(rng, 3, 3001, dtype)
            s = _exact_score(a, b, t, beta, dtype, src)
            assert oracle.fused_argmax_src(a, b, t, beta, src) == int(np.argmax(s))
    # the default source is the method's a - b
    a, b, t = _rows(rng, 3, 500, gen.F32)
    assert oracle.fused_argmax_src(a, b, t, 1.0, 0) == oracle.fused_argmax(a, b, t, 1.0)
