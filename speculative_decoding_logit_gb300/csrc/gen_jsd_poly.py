"""Build step: fit the polynomials the kernels use for the per-entry
Jensen-Shannon term, and write jsd_poly.inc.

For one vocabulary entry with probabilities p (first distribution) and
q = p * e^u (second), the entry's share of
    2 * JSD = sum_k [ p_k ln(2 p_k / (p_k + q_k)) + q_k ln(2 q_k / (p_k + q_k)) ]
is p * f(u) with
    f(u) = (1 + e^u) ln(2 / (1 + e^u)) + u e^u      (f >= 0, f(0) = 0, f ~ u^2/4).
The share is symmetric in p and q, so p f(u) = q f(-u), i.e. f(u) = e^u f(-u).

Narrow form (|u| <= U0): p f(u) = sqrt(p q) * u^2 * R(u^2).  R(u^2) = e^(-u/2) f(u) / u^2
is even in u (the symmetry above), so it is a polynomial in s = u^2 of low degree.
Writing the share this way keeps it exactly 0 at u = 0, so identical rows give a
divergence of exactly 0, and sqrt(p q) = exp((ln p + ln q) / 2) costs one exponential.

Wide form (any u): with m = max(p, q), s = |u| and r = e^-s = min(p,q)/max(p,q),
the entry's share is m * (A(r) - s*r) with A(r) = (1 + r) ln(2 / (1 + r)), and
A(r) = (1 - r) * B(r) with B smooth on [0, 1] (B(0) = ln 2, B(1) = 1).

A second, shorter narrow form (|u| <= U1 = 3, R of degree DEG1 = 6) serves pairs whose u stays
small (the AsymSpec pair a, b).  The degrees are the lowest that keep both narrow forms within
about 1.6e-7 relative in fp32, the size of ex2.approx's own error on the weights: the per-entry
term is bound by the fp32 pipe, so every multiply-add counts.

Both R and B are fitted here in 50-digit arithmetic by least squares in
relative error on Chebyshev nodes; coefficients are rounded to fp32 one at a
time from the highest degree down, each rounding followed by a refit of the
remaining lower coefficients.

Run:  python gen_jsd_poly.py   (rewrites jsd_poly.inc beside this file)
"""
import os
import struct

import mpmath as mp
import numpy as np

mp.mp.dps = 50
U0 = 4.0
DEG = 8  # degree of R in s = u^2
U1 = 3.0
DEG1 = 6  # degree of the short form's R


def f(u):
    u = mp.mpf(u)
    e = mp.e ** u
    return (1 + e) * mp.log(2 / (1 + e)) + u * e


def P(u):
    u = mp.mpf(u)
    if abs(u) < mp.mpf("1e-12"):
        return mp.mpf(1) / 4
    return f(u) / (u * u)


def Rfun(s):
    """R(s) = e^(-u/2) f(u) / u^2 at u = sqrt(s) (the same value at u = -sqrt(s))."""
    s = mp.mpf(s)
    if s < mp.mpf("1e-24"):
        return mp.mpf(1) / 4
    u = mp.sqrt(s)
    return P(u) * mp.e ** (-u / 2)


R_DEG = 11


def Bfun(r):
    r = mp.mpf(r)
    if abs(1 - r) < mp.mpf("1e-20"):
        return mp.mpf(1)
    return (1 + r) * mp.log(2 / (1 + r)) / (1 - r)


def f32(x):
    return float(np.float32(float(x)))


def fit(fixed, fun=None, deg=DEG, lo=-U0, hi=U0):
    """Least squares in relative error on Chebyshev nodes of [lo, hi] for the free
    (lower) coefficients, the ones in `fixed` (degree -> value) held."""
    fun = fun or P
    n = 8 * deg
    mid, half = (mp.mpf(hi) + lo) / 2, (mp.mpf(hi) - lo) / 2
    xs = [mid + half * mp.cos(mp.pi * (k + mp.mpf(1) / 2) / n) for k in range(n)]
    free = [d for d in range(deg + 1) if d not in fixed]
    A = mp.matrix(n, len(free))
    rhs = mp.matrix(n, 1)
    for i, x in enumerate(xs):
        w = 1 / fun(x)
        r = fun(x) - sum(fixed[d] * x ** d for d in fixed)
        rhs[i] = r * w
        for j, d in enumerate(free):
            A[i, j] = x ** d * w
    sol = mp.lu_solve(A.T * A, A.T * rhs)
    c = dict(fixed)
    for j, d in enumerate(free):
        c[d] = sol[j]
    return c


def fit_rounded(fun, deg, lo, hi):
    fixed = {}
    for d in range(deg, -1, -1):
        c = fit(fixed, fun, deg, lo, hi)
        fixed[d] = mp.mpf(f32(c[d]))
    return [float(fixed[d]) for d in range(deg + 1)]


def horner32(coef, xs32):
    acc = np.full_like(xs32, np.float32(coef[-1]))
    for d in range(len(coef) - 2, -1, -1):
        acc = (acc.astype(np.float64) * xs32 + np.float32(coef[d])).astype(np.float32)
    return acc


def emit(fh, name, var, coef):
    deg = len(coef) - 1
    fh.write(f"static __device__ __forceinline__ float {name}(float {var}) {{\n")
    fh.write(f"  float acc = {float(coef[deg]).hex()}f;  // c{deg}\n")
    for d in range(deg - 1, -1, -1):
        fh.write(f"  acc = fmaf(acc, {var}, {float(coef[d]).hex()}f);  // c{d} = {coef[d]:.9e}\n")
    fh.write("  return acc;\n}\n")


def emit2(fh, name, var, coef):
    """Packed form: the same Horner steps on two lanes per instruction (fma.rn.f32x2)."""
    deg = len(coef) - 1
    fh.write(f"static __device__ __forceinline__ float2 {name}(float2 {var}) {{\n")
    fh.write(f"  float2 acc = make_float2({float(coef[deg]).hex()}f, {float(coef[deg]).hex()}f);  // c{deg}\n")
    for d in range(deg - 1, -1, -1):
        c = float(coef[d]).hex()
        fh.write(f"  acc = asv::ffma2(acc, {var}, make_float2({c}f, {c}f));  // c{d}\n")
    fh.write("  return acc;\n}\n")


def main():
    S0 = U0 * U0
    coef = fit_rounded(Rfun, DEG, 0.0, S0)
    bcoef = fit_rounded(Bfun, R_DEG, 0.0, 1.0)
    rs = np.linspace(0, 1, 2001)
    berr = float(max(abs(sum(mp.mpf(bcoef[d]) * mp.mpf(x) ** d for d in range(R_DEG + 1)) / Bfun(x) - 1) for x in rs))
    rs32 = rs.astype(np.float32)
    bacc = horner32(bcoef, rs32)
    berr32 = float(max(abs(float(bacc[i]) / float(Bfun(float(rs32[i]))) - 1) for i in range(len(rs))))
    # exact-arithmetic relative error of R with the fp32 coefficients
    xs = np.linspace(0.0, S0, 4001)
    err = float(max(abs(sum(mp.mpf(coef[d]) * mp.mpf(x) ** d for d in range(DEG + 1)) / Rfun(x) - 1) for x in xs))
    # fp32 Horner evaluation, as the kernel does it
    xs32 = xs.astype(np.float32)
    acc = horner32(coef, xs32)
    err32 = float(max(abs(float(acc[i]) / float(Rfun(float(xs32[i]))) - 1) for i in range(len(xs))))
    S1 = U1 * U1
    coef1 = fit_rounded(Rfun, DEG1, 0.0, S1)
    xs1 = np.linspace(0.0, S1, 4001)
    err1 = float(max(abs(sum(mp.mpf(coef1[d]) * mp.mpf(x) ** d for d in range(DEG1 + 1)) / Rfun(x) - 1) for x in xs1))
    xs1_32 = xs1.astype(np.float32)
    acc1 = horner32(coef1, xs1_32)
    err1_32 = float(max(abs(float(acc1[i]) / float(Rfun(float(xs1_32[i]))) - 1) for i in range(len(xs1))))
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "jsd_poly.inc")
    with open(out, "w") as fh:
        fh.write("// Generated by gen_jsd_poly.py -- do not edit.\n")
        fh.write(f"// Narrow form: p f(u) = sqrt(p q) u^2 R(u^2) on |u| <= {U0}, R of degree {DEG} in u^2.\n")
        fh.write(f"//   max relative error of R: {err:.3e} (exact arithmetic), {err32:.3e} (fp32 Horner).\n")
        fh.write(f"// Wide form: A(r) = (1 - r) * B(r) on [0, 1], B of degree {R_DEG}.\n")
        fh.write(f"//   max relative error of B: {berr:.3e} (exact arithmetic), {berr32:.3e} (fp32 Horner).\n")
        fh.write(f"// Short narrow form: |u| <= {U1}, R of degree {DEG1} in u^2.\n")
        fh.write(f"//   max relative error of R: {err1:.3e} (exact arithmetic), {err1_32:.3e} (fp32 Horner).\n")
        fh.write(f"#define ASV_JSD_EVEN_S0 {S0:.1f}f\n")
        fh.write(f"#define ASV_JSD_SHORT_S0 {S1:.1f}f\n")
        emit(fh, "asv_jsd_even", "s", coef)
        emit(fh, "asv_jsd_wide_b", "r", bcoef)
        emit2(fh, "asv_jsd_even2", "s", coef)
        emit2(fh, "asv_jsd_wide_b2", "r", bcoef)
        emit2(fh, "asv_jsd_short2", "s", coef1)
    print(f"wrote {out}: R rel err {err:.3e} exact, {err32:.3e} fp32; B rel err {berr:.3e} exact, {berr32:.3e} fp32; "
          f"short R rel err {err1:.3e} exact, {err1_32:.3e} fp32")


if __name__ == "__main__":
    main()
