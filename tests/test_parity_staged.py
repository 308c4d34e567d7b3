"""GPU parity of the staged kernel (selected with set_kernel(KERNEL_STAGED): one CTA per SM, rows
cut into units staged in shared memory, partials exchanged through the workspace) against the
oracle and against the cluster kernel on the same inputs ("AsymSpec: Context-Asymmetric Speculative Decoding for Agentic LLMs", sec. 4.1-4.2
and 5; "E2-SCI: Elastic Edge-Cloud Speculative Decoding via Credit Inertia", Key design 3).  The
shapes cut rows into several units with a short last unit, and batches whose rows straddle two
steps of the CTAs' unit sequences."""
import numpy as np
import pytest
import torch

import gen
import oracle
from parity_util import compare_asymspec, to_device, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def asv():
    import speculative_decoding_logit_gb300 as m
    m.build()
    m.set_kernel(m.KERNEL_STAGED)
    yield m
    m.set_kernel(m.KERNEL_DEFAULT)


def _dev(batch):
    return (to_device(batch.a, batch.dtype), to_device(batch.b, batch.dtype), to_device(batch.t, batch.dtype),
            torch.from_numpy(batch.drafts).cuda())


class cluster_kernel:
    """Selects the cluster kernel for the calls inside."""

    def __init__(self, asv):
        self.asv = asv

    def __enter__(self):
        self.asv.set_kernel(self.asv.KERNEL_CLUSTER)

    def __exit__(self, *exc):
        self.asv.set_kernel(self.asv.KERNEL_STAGED)


@pytest.mark.parametrize("dtype,B,K,V", [(gen.BF16, 11, 2, 151936), (gen.F32, 7, 4, 151936), (gen.F32, 1, 2, 32000),
                                         (gen.BF16, 37, 3, 20000), (gen.F32, 13, 1, 4096), (gen.BF16, 5, 0, 8)])
def test_staged_asymspec_matches_oracle_and_cluster(asv, dtype, B, K, V):
    batch = gen.make_asymspec_batch("spiky", 500 + V + B, B, K, V, dtype, identical_frac=0.3)
    a, b, t, d = _dev(batch)
    plan = asv.query_plan(asv.ASV_MODE_ASYMSPEC, B, K, V, dtype)
    assert plan["bulk"] == 2, plan
    for beta, gamma in [(1.0, 0.5), (0.0, 1.0), (2.0, 0.4)]:
        out = asv.asymspec_verify(a, b, t, d, beta, gamma)
        torch.cuda.synchronize()
        ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, beta, gamma)
        compare_asymspec(out, ref, dtype)
        assert np.all(out.D.cpu().numpy()[batch.identical] == 0.0)
        with cluster_kernel(asv):
            cl = asv.asymspec_verify(a, b, t, d, beta, gamma)
            torch.cuda.synchronize()
        assert torch.equal(out.accept_len, cl.accept_len) and torch.equal(out.tokens, cl.tokens)
        assert torch.equal(out.req_status, cl.req_status)
        assert torch.allclose(out.D, cl.D, atol=tol(dtype), rtol=0)


@pytest.mark.parametrize("src", [1, 2])
def test_staged_delta_sources(asv, src):
    batch = gen.make_asymspec_batch("gumbel_zipf", 70 + src, 9, 3, 40000, gen.BF16)
    a, b, t, d = _dev(batch)
    out = asv.asymspec_verify(a, b, t, d, 1.5, 0.5, delta_source=src)
    torch.cuda.synchronize()
    ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.5, 0.5, delta_source=src)
    compare_asymspec(out, ref, gen.BF16)


@pytest.mark.parametrize("dtype,V", [(gen.BF16, 151936), (gen.F32, 30000)])
def test_staged_sci_windows(asv, dtype, V):
    B, K = 10, 8
    r0 = np.random.default_rng(V).uniform(0.0, 1.0, B)
    r_gpu = torch.from_numpy(r0.copy()).cuda()
    r_ref = r0.copy()
    p = asv.SciParams(alpha_omega=1.0)
    op = oracle.SciParams(p.T_base, p.alpha_omega, p.tau_credit, p.T_min, p.T_max, p.ewma_beta)
    for win in range(3):
        batch = gen.make_asymspec_batch("spiky", 800 + V + win, B, K, V, dtype)
        out = asv.sci_verify(to_device(batch.a, dtype), to_device(batch.t, dtype), torch.from_numpy(batch.drafts).cuda(),
                             r_gpu, p)
        torch.cuda.synchronize()
        ref = oracle.sci_verify(batch.a, batch.t, batch.drafts, r_ref, op)
        ok = (ref.flags & oracle.FLAGS_UNGRADED) == 0
        np.testing.assert_array_equal(out.accept_len.cpu().numpy()[ok], ref.accept_len[ok])
        np.testing.assert_array_equal(out.tokens.cpu().numpy()[ok], ref.tokens[ok])
        np.testing.assert_allclose(out.jsd.cpu().numpy(), ref.jsd, atol=tol(dtype), rtol=0)
        np.testing.assert_allclose(r_gpu.cpu().numpy()[ok], ref.r_hat[ok], atol=1e-15, rtol=0)
        r_gpu.copy_(torch.from_numpy(ref.r_hat))
        r_ref = ref.r_hat


@pytest.mark.parametrize("dtype,V", [(gen.BF16, 151936), (gen.F32, 9000)])
def test_staged_fused_and_sweep(asv, dtype, V):
    B, K = 6, 4
    batch = gen.make_asymspec_batch("spiky", 900 + V, B, K, V, dtype, identical_frac=0.3)
    a, b, t, d = _dev(batch)
    r0 = np.full(B, 0.6)
    r_gpu = torch.from_numpy(r0.copy()).cuda()
    out = asv.asymspec_sci_verify(a, b, t, d, 1.0, 0.5, r_gpu)
    torch.cuda.synchronize()
    ref_a = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.0, 0.5)
    ref_s = oracle.sci_verify(batch.a, batch.t, batch.drafts, r0)
    compare_asymspec(out, ref_a, dtype)
    ok = (ref_s.flags & oracle.FLAGS_UNGRADED) == 0
    np.testing.assert_array_equal(out.sci_accept_len.cpu().numpy()[ok], ref_s.accept_len[ok])
    np.testing.assert_array_equal(out.sci_tokens.cpu().numpy()[ok], ref_s.tokens[ok])
    np.testing.assert_allclose(out.jsd.cpu().numpy(), ref_s.jsd, atol=tol(dtype), rtol=0)
    betas, gammas = [0.0, 1.0, 1.5, 2.0], [0.4, 0.5, 0.7, 1.0]
    sw = asv.asymspec_verify_sweep(a, b, t, d, betas, gammas)
    torch.cuda.synchronize()
    for i, be in enumerate(betas):
        for j, ga in enumerate(gammas):
            ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, be, ga)
            ok = (ref.flags & oracle.FLAGS_UNGRADED) == 0
            np.testing.assert_array_equal(sw.accept_len[j].cpu().numpy()[ok], ref.accept_len[ok])
            np.testing.assert_array_equal(sw.tokens[i, j].cpu().numpy()[ok], ref.tokens[ok])


def test_staged_workspace_left_zeroed(asv):
    """Calls of every staged mode, of growing size, share one workspace and leave it zero: the
    exchange area's counters and partials are cleared by each row's finaliser."""
    shapes = [(3, 2, 151936, gen.BF16), (40, 3, 8192, gen.F32), (2, 8, 151936, gen.F32)]
    need = max(asv.workspace_bytes(m, B, K, V, dt) for B, K, V, dt in shapes
               for m in (asv.ASV_MODE_ASYMSPEC, asv.ASV_MODE_SCI, asv.ASV_MODE_SWEEP, asv.ASV_MODE_ASYMSPEC_SCI))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for B, K, V, dt in shapes:
        batch = gen.make_asymspec_batch("spiky", 60 + B, B, K, V, dt)
        a, b, t, d = _dev(batch)
        r = torch.full((B,), 0.6, dtype=torch.float64, device="cuda")
        asv.asymspec_verify(a, b, t, d, 1.0, 0.5, workspace=ws)
        asv.sci_verify(a, t, d, r, workspace=ws)
        asv.asymspec_verify_sweep(a, b, t, d, [0.0, 1.0], [0.5], workspace=ws)
        asv.asymspec_sci_verify(a, b, t, d, 1.0, 0.5, r, workspace=ws)
        torch.cuda.synchronize()
        assert int(torch.count_nonzero(ws)) == 0, (B, K, V)
