"""Every request of the large workloads graded against the oracle, at full size, in the launch
configuration the benchmark uses:

  * the 256 x 5 x 151936 fp32 AsymSpec sweep (30 % of requests with a == b): all 16 (beta, gamma)
    points as single-outcome launches and from the one-read sweep kernel
    ("AsymSpec: Context-Asymmetric Speculative Decoding for Agentic LLMs", sec. 4.1-4.2, sec. 5);
  * the 1024 x 9 x 151936 bf16 batch: plain AsymSpec, AsymSpec fused with one E2-SCI window over
    two windows, and five sequential E2-SCI windows with the credit state carried on the device
    ("E2-SCI: Elastic Edge-Cloud Speculative Decoding via Credit Inertia", Key designs 1 and 3).

Requests the oracle flags (gate margin or threshold within 1e-6, or an argmax within
single-precision rounding of another entry) are counted, not graded; D, log-sum-exps and JSD are
compared on every finite row.  The oracle runs over the host cores in spawned processes."""
import numpy as np
import pytest
import torch

import gen
import oracle
from full_grading import Tally, compare_requests, grade_asymspec_batch, grade_sci_window, host_pool
from parity_util import to_device, tol

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

BETAS = [0.0, 1.0, 1.5, 2.0]
GAMMAS = [0.4, 0.5, 0.7, 1.0]


@pytest.fixture(scope="module")
def asv():
    import speculative_decoding_logit_gb300 as m
    m.build()
    return m


@pytest.fixture(scope="module")
def pool():
    p = host_pool()
    yield p
    p.close()
    p.join()


def _np(x):
    return x.cpu().numpy()


def _close_on_finite(gpu, ref, flags, atol, what):
    fin = (flags & 1) == 0
    np.testing.assert_allclose(gpu[fin], ref[fin], atol=atol, rtol=0, err_msg=what)


def _report(name, tally, differs=None):
    msg = f"{name}: {tally.graded} requests graded bit-exact, {tally.flagged} flagged"
    if differs is not None:
        msg += f"; rows where a single-precision argmax differs from the exact one: {differs[0]} (all near ties)"
    print(msg)


def test_sweep_b256_k4_v151936_f32_every_request(asv, pool):
    w = gen.WORKLOADS["asymspec_sweep_b256_k4_v151936_f32"]
    runs = [tuple(r) for r in w.params["runs"]]
    g = grade_asymspec_batch(pool, w, runs)
    assert g.identical.sum() == round(0.3 * w.B)
    a, b, t = (to_device(x, w.dtype) for x in (g.a, g.b, g.t))
    d = torch.from_numpy(g.drafts).cuda()
    tally = Tally()
    for (beta, gamma), ref, differs in zip(runs, g.refs, g.fp32_differs):
        assert differs[1] == differs[0], "a single-precision winner differs on a row not marked near"
        out = asv.asymspec_verify(a, b, t, d, beta, gamma)
        torch.cuda.synchronize()
        what = f"beta {beta} gamma {gamma}"
        compare_requests(_np(out.accept_len), _np(out.tokens), _np(out.req_status).astype(np.uint32),
                         ref.accept_len, ref.tokens, ref.flags, tally, what)
        D = _np(out.D).astype(np.float64)
        _close_on_finite(D, ref.D, ref.flags, tol(w.dtype), what)
        _close_on_finite(_np(out.lse).astype(np.float64), ref.lse, ref.flags, tol(w.dtype), what)
        assert np.all(D[g.identical] == 0.0)
    _report("single-outcome launches", tally, g.fp32_differs[0])
    # The one-read sweep kernel: every grid point from one launch.
    out = asv.asymspec_verify_sweep(a, b, t, d, BETAS, GAMMAS)
    torch.cuda.synchronize()
    acc, tok, st = _np(out.accept_len), _np(out.tokens), _np(out.req_status).astype(np.uint32)
    sweep = Tally()
    for i, beta in enumerate(BETAS):
        for j, gamma in enumerate(GAMMAS):
            ref = g.refs[runs.index((beta, gamma))]
            compare_requests(acc[j], tok[i, j], st, ref.accept_len, ref.tokens, ref.flags, sweep,
                             f"sweep point beta {beta} gamma {gamma}")
    _close_on_finite(_np(out.D).astype(np.float64), g.refs[0].D, g.refs[0].flags, tol(w.dtype), "sweep D")
    _report("sweep kernel", sweep)
    total = tally.graded + tally.flagged
    assert tally.flagged <= 0.05 * total and sweep.flagged == tally.flagged


def test_asymspec_b1024_k8_v151936_every_request(asv, pool):
    w = gen.WORKLOADS["sci_asymspec_b1024_k8_v151936_bf16"]
    g = grade_asymspec_batch(pool, w, [(1.0, 0.5)], seed=w.seed + 11)
    a, b, t = (to_device(x, w.dtype) for x in (g.a, g.b, g.t))
    d = torch.from_numpy(g.drafts).cuda()
    out = asv.asymspec_verify(a, b, t, d, 1.0, 0.5)
    torch.cuda.synchronize()
    ref = g.refs[0]
    tally = Tally()
    compare_requests(_np(out.accept_len), _np(out.tokens), _np(out.req_status).astype(np.uint32), ref.accept_len,
                     ref.tokens, ref.flags, tally, "AsymSpec 1024 x 9")
    _close_on_finite(_np(out.D).astype(np.float64), ref.D, ref.flags, tol(w.dtype), "D")
    _close_on_finite(_np(out.lse).astype(np.float64), ref.lse, ref.flags, tol(w.dtype), "lse")
    assert g.fp32_differs[0][1] == g.fp32_differs[0][0]
    _report("AsymSpec 1024 x 9 x 151936 bf16", tally, g.fp32_differs[0])
    assert tally.flagged <= 0.05 * w.B


def test_fused_b1024_k8_v151936_two_windows_every_request(asv, pool):
    """AsymSpec fused with an E2-SCI window, two windows, credit state carried on the device."""
    w = gen.WORKLOADS["sci_asymspec_b1024_k8_v151936_bf16"]
    r_ref = np.full(w.B, w.params["r_hat0"])
    r_gpu = torch.from_numpy(r_ref.copy()).cuda()
    ta, ts = Tally(), Tally()
    for win in range(2):
        g = grade_asymspec_batch(pool, w, [(1.0, 0.5)], seed=w.seed + 20 + win, sci_r_hat=r_ref)
        a, b, t = (to_device(x, w.dtype) for x in (g.a, g.b, g.t))
        d = torch.from_numpy(g.drafts).cuda()
        out = asv.asymspec_sci_verify(a, b, t, d, 1.0, 0.5, r_gpu)
        torch.cuda.synchronize()
        ref_a, ref_s = g.refs[0], g.sci
        st = _np(out.req_status).astype(np.uint32)
        compare_requests(_np(out.accept_len), _np(out.tokens), st, ref_a.accept_len, ref_a.tokens, ref_a.flags, ta,
                         f"fused window {win}: AsymSpec")
        compare_requests(_np(out.sci_accept_len), _np(out.sci_tokens), st, ref_s.accept_len, ref_s.tokens,
                         ref_s.flags, ts, f"fused window {win}: E2-SCI")
        _close_on_finite(_np(out.D).astype(np.float64), ref_a.D, ref_a.flags, tol(w.dtype), "D")
        _close_on_finite(_np(out.jsd).astype(np.float64), ref_s.jsd, ref_s.flags, tol(w.dtype), "J")
        np.testing.assert_allclose(_np(out.T), ref_s.T, atol=1e-7)
        r_new = _np(r_gpu)
        ok = (ref_s.flags & oracle.FLAGS_UNGRADED) == 0
        np.testing.assert_allclose(r_new[ok], ref_s.r_hat[ok], atol=1e-15, rtol=0)
        # flagged requests continue from the oracle's state on both sides
        r_gpu.copy_(torch.from_numpy(ref_s.r_hat))
        r_ref = ref_s.r_hat
        del a, b, t
    _report("fused AsymSpec", ta)
    _report("fused E2-SCI", ts)
    assert ta.flagged <= 0.05 * 2 * w.B and ts.flagged <= 0.05 * 2 * w.B


def test_sci_b1024_k8_v151936_five_windows_every_request(asv, pool):
    """k = 5 windows, each with its own seeded tensors, credit state carried on the device
    (E2-SCI Key design 1: history of k = 5 windows; Key design 3: EWMA credit, clamped threshold)."""
    w = gen.WORKLOADS["sci_asymspec_b1024_k8_v151936_bf16"]
    r_ref = np.full(w.B, w.params["r_hat0"])
    r_gpu = torch.from_numpy(r_ref.copy()).cuda()
    tally = Tally()
    for win in range(w.params["windows"]):
        a_h, t_h, d_h, ref = grade_sci_window(pool, w, w.seed + win, r_ref)
        a, t = to_device(a_h, w.dtype), to_device(t_h, w.dtype)
        out = asv.sci_verify(a, t, torch.from_numpy(d_h).cuda(), r_gpu)
        torch.cuda.synchronize()
        compare_requests(_np(out.accept_len), _np(out.tokens), _np(out.req_status).astype(np.uint32),
                         ref.accept_len, ref.tokens, ref.flags, tally, f"E2-SCI window {win}")
        _close_on_finite(_np(out.jsd).astype(np.float64), ref.jsd, ref.flags, tol(w.dtype), "J")
        np.testing.assert_allclose(_np(out.T), ref.T, atol=1e-7)
        ok = (ref.flags & oracle.FLAGS_UNGRADED) == 0
        np.testing.assert_allclose(_np(r_gpu)[ok], ref.r_hat[ok], atol=1e-15, rtol=0)
        r_gpu.copy_(torch.from_numpy(ref.r_hat))
        r_ref = ref.r_hat
        del a, t
    _report("E2-SCI five windows", tally)
    assert tally.flagged <= 0.05 * 5 * w.B
