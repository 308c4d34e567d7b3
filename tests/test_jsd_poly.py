"""The fitted polynomials the kernels evaluate for the per-entry Jensen-Shannon term
(speculative_decoding_logit_gb300/csrc/jsd_poly.inc), pinned to the mathematics they stand for.

For one vocabulary entry with probabilities p and q = p e^u, the entry's share of 2 JSD is
p f(u), f(u) = (1 + e^u) ln(2 / (1 + e^u)) + u e^u ("AsymSpec: Context-Asymmetric Speculative
Decoding for Agentic LLMs", sec. 4.2: D = JSD(softmax a || softmax b), natural log, weights 1/2).
The narrow forms write it as sqrt(p q) u^2 R(u^2), R(s) = e^(-u/2) f(u) / u^2 at u = sqrt(s); the
wide form as max(p, q) ((1 - r) B(r) - |u| r), r = e^-|u|, B(r) = (1 + r) ln(2 / (1 + r)) / (1 - r).
The table's coefficients are evaluated here with fp32 Horner steps (one rounding per step, as the
kernels' fused multiply-adds do) and compared with R and B computed in 40-digit arithmetic; then the
narrow form, assembled as the kernel assembles it, reproduces scipy's Jensen-Shannon divergence."""
import os
import re

import numpy as np
import pytest

mp = pytest.importorskip("mpmath")
spd = pytest.importorskip("scipy.spatial.distance")

INC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "speculative_decoding_logit_gb300", "csrc", "jsd_poly.inc")


def _table():
    text = open(INC).read()
    s0 = {m.group(1): float(m.group(2)) for m in re.finditer(r"#define (ASV_JSD_\w+_S0) ([0-9.]+)f", text)}
    polys = {}
    for m in re.finditer(r"static __device__ __forceinline__ (float2?) (\w+)\(float2? \w+\) \{(.*?)\n\}", text, re.S):
        hexes = [float.fromhex(h) for h in re.findall(r"(-?0x[0-9a-fA-F.p+-]+)f", m.group(3))]
        if m.group(1) == "float2":  # packed form: every constant is given once per lane
            assert hexes[0::2] == hexes[1::2]
            hexes = hexes[0::2]
        # the leading coefficient first, then one per Horner step (highest degree first)
        polys[m.group(2)] = hexes
    return s0, polys


def _horner32(coef_high_first, x):
    x = np.asarray(x, np.float32).astype(np.float64)
    acc = np.full(x.shape, np.float32(coef_high_first[0]))
    for c in coef_high_first[1:]:
        acc = (acc.astype(np.float64) * x + np.float64(np.float32(c))).astype(np.float32)
    return acc.astype(np.float64)


mp.mp.dps = 40


def _R(s):
    s = mp.mpf(s)
    if s == 0:
        return mp.mpf(1) / 4
    u = mp.sqrt(s)
    e = mp.e ** u
    f = (1 + e) * mp.log(2 / (1 + e)) + u * e
    return mp.e ** (-u / 2) * f / s


def _B(r):
    r = mp.mpf(r)
    if r == 1:
        return mp.mpf(1)
    return (1 + r) * mp.log(2 / (1 + r)) / (1 - r)


def test_table_domains():
    s0, polys = _table()
    assert s0["ASV_JSD_EVEN_S0"] == 16.0 and s0["ASV_JSD_SHORT_S0"] == 9.0
    assert {"asv_jsd_even", "asv_jsd_even2", "asv_jsd_short2", "asv_jsd_wide_b", "asv_jsd_wide_b2"} <= set(polys)
    # the packed forms carry the scalar forms' coefficients
    assert polys["asv_jsd_even2"] == polys["asv_jsd_even"]
    assert polys["asv_jsd_wide_b2"] == polys["asv_jsd_wide_b"]
    # the short form is the shorter one
    assert len(polys["asv_jsd_short2"]) < len(polys["asv_jsd_even"])


@pytest.mark.parametrize("name,S0", [("asv_jsd_even", 16.0), ("asv_jsd_short2", 9.0)])
def test_narrow_forms_against_R(name, S0):
    _, polys = _table()
    coef = polys[name]
    s = np.concatenate([np.linspace(0.0, S0, 1201), [1e-6, 1e-3, S0]]).astype(np.float32)
    got = _horner32(coef, s)
    ref = np.array([float(_R(float(x))) for x in s])
    assert np.max(np.abs(got / ref - 1.0)) < 2.0e-7


def test_wide_form_against_B():
    _, polys = _table()
    r = np.concatenate([np.linspace(0.0, 1.0, 1001), [1e-7, 0.999999]]).astype(np.float32)
    got = _horner32(polys["asv_jsd_wide_b"], r)
    ref = np.array([float(_B(float(x))) for x in r])
    assert np.max(np.abs(got / ref - 1.0)) < 1.0e-7


@pytest.mark.parametrize("name,umax", [("asv_jsd_short2", 3.0), ("asv_jsd_even", 4.0)])
def test_narrow_form_reproduces_scipy_jsd(name, umax):
    """D = 1/2 sum sqrt(p q) u^2 R(u^2) with u = ln q - ln p inside the form's domain, against
    scipy's Jensen-Shannon distance squared (natural log)."""
    _, polys = _table()
    coef = polys[name]
    rng = np.random.default_rng(1234)
    for _ in range(20):
        n = 64
        lp = rng.normal(0.0, 2.0, n)
        p = np.exp(lp - lp.max())
        p /= p.sum()
        # q = p e^w / Z: u = w - ln Z with |ln Z| <= max |w|, so |w| <= umax / 2 keeps |u| <= umax
        q = p * np.exp(rng.uniform(-0.499 * umax, 0.499 * umax, n))
        q /= q.sum()
        u = np.log(q) - np.log(p)
        assert np.all(np.abs(u) <= umax)
        R = _horner32(coef, (u * u).astype(np.float32))
        D = 0.5 * np.sum(np.sqrt(p * q) * u * u * R)
        ref = spd.jensenshannon(p, q) ** 2
        assert abs(D - ref) <= 3e-7 * ref + 1e-12
