"""GPU parity at the extremes of the shapes: more drafts per request than one 32-row step of the
last-arriver scan (the accepted prefix ending before, at and after the step boundary, and every
draft accepted), in every mode, and vocabularies larger than the workloads' (2^18 entries, and an
odd length that takes the element-wise path).  Decisions and tokens bit-exact against the oracle
(flagged requests counted, not graded), numeric fields within the usual tolerance."""
import numpy as np
import pytest
import scipy.special as sps
import torch

import gen
import oracle
from parity_util import compare_asymspec, to_device, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def asv():
    import speculative_decoding_logit_gb300 as m
    m.build()
    return m


# First rejection position per request (K means every draft is accepted).
STOPS = [0, 30, 31, 32, 33, 39, 40]
K_LONG = 40


def _forced_asymspec(seed, V):
    """fp32 rows where request r's gate passes for drafts before STOPS[r] and fails at STOPS[r]:
    the draft token's verifier logit is raised by 12 (accept) or lowered by 12 (reject)."""
    B = len(STOPS)
    batch = gen.make_asymspec_batch("spiky", seed, B, K_LONG, V, gen.F32)
    a, b, t = batch.a.copy(), batch.b.copy(), batch.t.copy()
    d = batch.drafts
    for r, n in enumerate(STOPS):
        for i in range(K_LONG):
            if i < n:
                t[r, i, d[r, i]] += 12.0
            elif i == n:
                t[r, i, d[r, i]] -= 12.0
    return a, b, t, d


def test_asymspec_long_draft_runs(asv):
    a, b, t, d = _forced_asymspec(8101, 2048)
    out = asv.asymspec_verify(to_device(a, gen.F32), to_device(b, gen.F32), to_device(t, gen.F32),
                              torch.from_numpy(d).cuda(), 1.0, 0.5)
    torch.cuda.synchronize()
    ref = oracle.asymspec_verify(a, b, t, d, 1.0, 0.5)
    compare_asymspec(out, ref, gen.F32)
    np.testing.assert_array_equal(out.accept_len.cpu().numpy(), np.minimum(STOPS, K_LONG))


def test_sweep_long_draft_runs(asv):
    a, b, t, d = _forced_asymspec(8102, 2048)
    betas, gammas = [0.0, 1.0, 2.0], [0.3, 0.5, 1.0]
    out = asv.asymspec_verify_sweep(to_device(a, gen.F32), to_device(b, gen.F32), to_device(t, gen.F32),
                                    torch.from_numpy(d).cuda(), betas, gammas)
    torch.cuda.synchronize()
    for i, beta in enumerate(betas):
        for g, gamma in enumerate(gammas):
            ref = oracle.asymspec_verify(a, b, t, d, beta, gamma)
            for r in range(len(STOPS)):
                if ref.flags[r] & oracle.FLAGS_UNGRADED:
                    continue
                assert out.accept_len[g, r].item() == ref.accept_len[r]
                np.testing.assert_array_equal(out.tokens[i, g, r].cpu().numpy(), ref.tokens[r])


@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_sci_long_draft_runs(asv, dtype):
    """E2-SCI windows of 40 drafts: the target equals the draft distribution (J = 0, accepted) before
    the stop and differs strongly at it (J above any threshold the credit state gives)."""
    B, V = len(STOPS), 2048
    batch = gen.make_asymspec_batch("spiky", 8103, B, K_LONG, V, gen.F32)
    a = batch.a.copy()
    t = batch.t.copy()
    rng = np.random.default_rng(8103)
    for r, n in enumerate(STOPS):
        for i in range(K_LONG + 1):
            if i < n:
                t[r, i] = a[r, i]
            elif i == n:
                t[r, i] = a[r, i] + rng.normal(0.0, 8.0, V)
    a_s, t_s = gen.store(a, dtype), gen.store(t, dtype)
    r_hat = np.full(B, 0.6)
    r = torch.from_numpy(r_hat.copy()).cuda()
    out = asv.sci_verify(to_device(a_s, dtype), to_device(t_s, dtype), torch.from_numpy(batch.drafts).cuda(), r)
    torch.cuda.synchronize()
    ref = oracle.sci_verify(a_s, t_s, batch.drafts, r_hat)
    st = out.req_status.cpu().numpy().astype(np.uint32)
    np.testing.assert_array_equal(st & 3, ref.flags & 3)
    for q in range(B):
        if ref.flags[q] & oracle.FLAGS_UNGRADED:
            continue
        assert out.accept_len[q].item() == ref.accept_len[q] == min(STOPS[q], K_LONG)
        np.testing.assert_array_equal(out.tokens[q].cpu().numpy(), ref.tokens[q])
        assert r[q].item() == pytest.approx(ref.r_hat[q], abs=1e-15)
    np.testing.assert_allclose(out.jsd.cpu().numpy(), ref.jsd, atol=tol(dtype), rtol=0)


def test_rapid_long_draft_runs(asv):
    """RAPID with 40 drafts: q equals softmax(z) (eta = 0 makes the target p itself, so a draft is
    rejected only when u exceeds p/q, which is 1 up to rounding) except at each request's stop,
    where the draft's target logit is pushed down by 30 (p(d) ~ 0, certain rejection)."""
    B, G, V = len(STOPS), K_LONG, 2048
    rng = np.random.default_rng(8104)
    z = rng.normal(0.0, 2.0, (B, G + 1, V)).astype(np.float32)
    d = np.zeros((B, G), np.int32)
    for r in range(B):
        for i in range(G):
            d[r, i] = rng.integers(0, 8)  # among the first ids; their mass is what it is
    q = sps.softmax(z.astype(np.float64), axis=-1).astype(np.float32)
    for r, n in enumerate(STOPS):
        if n < G:
            z[r, n, d[r, n]] -= 30.0
    out = asv.rapid_verify(torch.from_numpy(z).cuda(), torch.from_numpy(q).cuda(), torch.from_numpy(d).cuda(),
                           1.0, 0.0, 0.1, 1234)
    torch.cuda.synchronize()
    ref = oracle.rapid_verify(z, q, d, 1.0, 0.0, 0.1, 1234)
    st = out.req_status.cpu().numpy().astype(np.uint32)
    np.testing.assert_array_equal(st & 3, ref.flags & 3)
    graded = 0
    for r in range(B):
        if ref.flags[r] & oracle.FLAGS_UNGRADED:
            continue
        graded += 1
        assert out.accept_len[r].item() == ref.accept_len[r]
        np.testing.assert_array_equal(out.tokens[r].cpu().numpy(), ref.tokens[r])
    assert graded >= B - 1
    assert max(ref.accept_len) >= 33  # some request's accepted prefix crosses the 32-row step


@pytest.mark.parametrize("dtype,V", [(gen.BF16, 262144), (gen.F32, 262147)])
def test_asymspec_large_vocabulary(asv, dtype, V):
    batch = gen.make_asymspec_batch("gumbel_zipf", 8200 + V, 2, 2, V, dtype)
    out = asv.asymspec_verify(to_device(batch.a, dtype), to_device(batch.b, dtype), to_device(batch.t, dtype),
                              torch.from_numpy(batch.drafts).cuda(), 1.0, 0.5)
    torch.cuda.synchronize()
    ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.0, 0.5)
    compare_asymspec(out, ref, dtype)


def test_sci_and_rapid_large_vocabulary(asv):
    V = 262144
    batch = gen.make_asymspec_batch("spiky", 8300, 2, 3, V, gen.BF16)
    r_hat = np.full(2, 0.6)
    r = torch.from_numpy(r_hat.copy()).cuda()
    out = asv.sci_verify(to_device(batch.a, gen.BF16), to_device(batch.t, gen.BF16),
                         torch.from_numpy(batch.drafts).cuda(), r)
    torch.cuda.synchronize()
    ref = oracle.sci_verify(batch.a, batch.t, batch.drafts, r_hat)
    for q in range(2):
        if not (ref.flags[q] & oracle.FLAGS_UNGRADED):
            assert out.accept_len[q].item() == ref.accept_len[q]
            np.testing.assert_array_equal(out.tokens[q].cpu().numpy(), ref.tokens[q])
    np.testing.assert_allclose(out.jsd.cpu().numpy(), ref.jsd, atol=tol(gen.BF16), rtol=0)

    rb = gen.make_rapid_batch(8301, 2, 3, V)
    out = asv.rapid_verify(torch.from_numpy(rb.z).cuda(), torch.from_numpy(rb.q).cuda(),
                           torch.from_numpy(rb.drafts).cuda(), 1.0, 10.0, 0.1, 1234)
    torch.cuda.synchronize()
    ref = oracle.rapid_verify(rb.z, rb.q, rb.drafts, 1.0, 10.0, 0.1, 1234)
    for q in range(2):
        if not (ref.flags[q] & oracle.FLAGS_UNGRADED):
            assert out.accept_len[q].item() == ref.accept_len[q]
            np.testing.assert_array_equal(out.tokens[q].cpu().numpy(), ref.tokens[q])
