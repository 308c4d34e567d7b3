"""GPU parity for the cluster-wide combination of a row's partials at every cluster size.  The row
statistics, the argmax slots and the pass-B sums of a row are read four CTAs at a time and combined
in rank order, moving the running sum to a new reference when a later group holds the larger
maximum; clusters of 5 to 16 CTAs take more than one group, some with a last group that is partly
empty.  Every mode of the AsymSpec / E2-SCI kernel is compared with the oracle at such sizes, and a
short vocabulary leaves some CTAs of a 16-CTA cluster without entries."""
import numpy as np
import pytest
import torch

import gen
import oracle
from parity_util import compare_asymspec, to_device, tol

pytestmark = pytest.mark.gpu

SIZES = [4, 5, 7, 12, 16]


@pytest.fixture(scope="module")
def asv():
    import speculative_decoding_logit_gb300 as m
    m.build()
    return m


class forced_cluster:
    def __init__(self, asv, c):
        self.asv, self.c = asv, c

    def __enter__(self):
        self.asv.set_tuning(self.c, 256)

    def __exit__(self, *exc):
        self.asv.set_tuning(0, 0)


def _dev(batch):
    return (to_device(batch.a, batch.dtype), to_device(batch.b, batch.dtype), to_device(batch.t, batch.dtype),
            torch.from_numpy(batch.drafts).cuda())


@pytest.mark.parametrize("cluster", SIZES)
@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_asymspec_every_group_size(asv, cluster, dtype):
    # spiky rows: the row maximum lands in a random CTA, so later groups often raise the reference
    batch = gen.make_asymspec_batch("spiky", 900 + cluster, 10, 3, 6000, dtype, identical_frac=0.2)
    with forced_cluster(asv, cluster):
        out = asv.asymspec_verify(*_dev(batch), 1.0, 0.5)
        torch.cuda.synchronize()
        assert asv.query_plan(asv.ASV_MODE_ASYMSPEC, 10, 3, 6000, 0 if dtype == gen.F32 else 1)["cluster"] == cluster
    ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.0, 0.5)
    compare_asymspec(out, ref, dtype)


@pytest.mark.parametrize("cluster", [5, 12, 16])
def test_sweep_every_group_size(asv, cluster):
    batch = gen.make_asymspec_batch("gumbel_zipf", 910 + cluster, 8, 3, 5000, gen.BF16)
    betas, gammas = [0.0, 1.0, 2.0], [0.4, 1.0]
    with forced_cluster(asv, cluster):
        out = asv.asymspec_verify_sweep(*_dev(batch), betas, gammas)
        torch.cuda.synchronize()
    for i, beta in enumerate(betas):
        for g, gamma in enumerate(gammas):
            ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, beta, gamma)
            for r in range(8):
                if ref.flags[r] & oracle.FLAGS_UNGRADED:
                    continue
                assert out.accept_len[g, r].item() == ref.accept_len[r]
                np.testing.assert_array_equal(out.tokens[i, g, r].cpu().numpy(), ref.tokens[r])
    fin = (ref.flags & 1) == 0
    np.testing.assert_allclose(out.D.cpu().numpy()[fin], ref.D[fin], atol=tol(gen.BF16), rtol=0)
    np.testing.assert_allclose(out.lse.cpu().numpy()[fin], ref.lse[fin], atol=tol(gen.BF16), rtol=0)


@pytest.mark.parametrize("cluster", [5, 16])
@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_sci_and_fused_every_group_size(asv, cluster, dtype):
    B, K, V = 8, 4, 7000
    batch = gen.make_asymspec_batch("spiky", 920 + cluster, B, K, V, dtype)
    r0 = np.random.default_rng(cluster).uniform(0.2, 1.0, B)
    a, b, t, d = _dev(batch)
    with forced_cluster(asv, cluster):
        r_sci = torch.from_numpy(r0.copy()).cuda()
        sci = asv.sci_verify(a, t, d, r_sci)
        r_fused = torch.from_numpy(r0.copy()).cuda()
        fused = asv.asymspec_sci_verify(a, b, t, d, 1.0, 0.5, r_fused)
        torch.cuda.synchronize()
    ref_s = oracle.sci_verify(batch.a, batch.t, batch.drafts, r0.copy())
    ref_a = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.0, 0.5)
    for q in range(B):
        if not (ref_s.flags[q] & oracle.FLAGS_UNGRADED):
            assert sci.accept_len[q].item() == ref_s.accept_len[q]
            np.testing.assert_array_equal(sci.tokens[q].cpu().numpy(), ref_s.tokens[q])
            assert fused.sci_accept_len[q].item() == ref_s.accept_len[q]
            np.testing.assert_array_equal(fused.sci_tokens[q].cpu().numpy(), ref_s.tokens[q])
            assert r_sci[q].item() == pytest.approx(ref_s.r_hat[q], abs=1e-15)
            assert r_fused[q].item() == pytest.approx(ref_s.r_hat[q], abs=1e-15)
        if not (ref_a.flags[q] & oracle.FLAGS_UNGRADED):
            assert fused.accept_len[q].item() == ref_a.accept_len[q]
            np.testing.assert_array_equal(fused.tokens[q].cpu().numpy(), ref_a.tokens[q])
    np.testing.assert_allclose(sci.jsd.cpu().numpy(), ref_s.jsd, atol=tol(dtype), rtol=0)
    np.testing.assert_allclose(fused.jsd.cpu().numpy(), ref_s.jsd, atol=tol(dtype), rtol=0)
    np.testing.assert_allclose(fused.D.cpu().numpy(), ref_a.D, atol=tol(dtype), rtol=0)


@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_short_vocabulary_leaves_ctas_empty(asv, dtype):
    """V = 100 over 16 CTAs: the slices of the last CTAs hold no entries (maximum -inf, sums 0)."""
    batch = gen.make_asymspec_batch("spiky", 930, 6, 2, 100, dtype, identical_frac=0.3)
    with forced_cluster(asv, 16):
        out = asv.asymspec_verify(*_dev(batch), 1.0, 0.5)
        torch.cuda.synchronize()
    ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.0, 0.5)
    compare_asymspec(out, ref, dtype)
