"""GPU parity for the one-read multi-outcome modes: the all-(beta, gamma) AsymSpec sweep
("AsymSpec: Context-Asymmetric Speculative Decoding for Agentic LLMs", sec. 5: beta and gamma over a
flat region) and AsymSpec fused with one E2-SCI window ("E2-SCI: Elastic Edge-Cloud Speculative
Decoding via Credit Inertia", Key design 3).  Every grid point / mode is compared with the oracle's
single-outcome result; requests the oracle flags are counted, not graded."""
import numpy as np
import pytest
import torch

import gen
import oracle
from parity_util import to_device, tol

pytestmark = pytest.mark.gpu

BETAS = [0.0, 1.0, 1.5, 2.0]
GAMMAS = [0.4, 0.5, 0.7, 1.0]


@pytest.fixture(scope="module")
def asv():
    import speculative_decoding_logit_gb300 as m
    m.build()
    return m


def _dev(batch):
    return (to_device(batch.a, batch.dtype), to_device(batch.b, batch.dtype), to_device(batch.t, batch.dtype),
            torch.from_numpy(batch.drafts).cuda())


@pytest.mark.parametrize("dtype,V", [(gen.F32, 4096), (gen.BF16, 6000), (gen.F32, 1001)])
def test_sweep_matches_every_grid_point(asv, dtype, V):
    batch = gen.make_asymspec_batch("spiky", 300 + V, 16, 4, V, dtype, identical_frac=0.3)
    a, b, t, d = _dev(batch)
    out = asv.asymspec_verify_sweep(a, b, t, d, BETAS, GAMMAS)
    torch.cuda.synchronize()
    acc = out.accept_len.cpu().numpy()
    tok = out.tokens.cpu().numpy()
    st = out.req_status.cpu().numpy().astype(np.uint32)
    graded = 0
    for i, be in enumerate(BETAS):
        for j, ga in enumerate(GAMMAS):
            ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, be, ga)
            np.testing.assert_array_equal(st & 3, ref.flags & 3)
            for r in range(16):
                if ref.flags[r] & oracle.FLAGS_UNGRADED:
                    continue
                graded += 1
                assert acc[j, r] == ref.accept_len[r], (be, ga, r)
                np.testing.assert_array_equal(tok[i, j, r], ref.tokens[r], err_msg=f"beta {be} gamma {ga} req {r}")
    assert graded >= 16 * 16 - 40
    fin = (ref.flags & 1) == 0
    np.testing.assert_allclose(out.D.cpu().numpy()[fin], ref.D[fin], atol=tol(dtype), rtol=0)
    np.testing.assert_allclose(out.lse.cpu().numpy()[fin], ref.lse[fin], atol=tol(dtype), rtol=0)
    # D and the log-sum-exps do not depend on (beta, gamma): the single-outcome kernel gives the same bits
    single = asv.asymspec_verify(a, b, t, d, 1.0, 0.5)
    torch.cuda.synchronize()
    assert torch.equal(single.D, out.D) and torch.equal(single.lse, out.lse)


def test_sweep_fewer_points_and_workspace(asv):
    batch = gen.make_asymspec_batch("gumbel_zipf", 77, 9, 3, 3000, gen.BF16)
    a, b, t, d = _dev(batch)
    need = asv.workspace_bytes(asv.ASV_MODE_SWEEP, 9, 3, 3000, asv.ASV_BF16)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    out = asv.asymspec_verify_sweep(a, b, t, d, [0.5, 2.0], [0.3], workspace=ws)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(ws)) == 0
    for i, be in enumerate([0.5, 2.0]):
        ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, be, 0.3)
        for r in range(9):
            if ref.flags[r] & oracle.FLAGS_UNGRADED:
                continue
            assert out.accept_len[0, r].item() == ref.accept_len[r]
            np.testing.assert_array_equal(out.tokens[i, 0, r].cpu().numpy(), ref.tokens[r])


@pytest.mark.parametrize("dtype,V", [(gen.BF16, 8192), (gen.F32, 4096), (gen.BF16, 1001)])
def test_fused_asymspec_and_sci(asv, dtype, V):
    w = gen.WORKLOADS["sci_asymspec_b1024_k8_v151936_bf16"]
    B, K = 16, 8
    r0 = np.random.default_rng(V).uniform(0.2, 1.0, B)
    r_gpu = torch.from_numpy(r0.copy()).cuda()
    r_ref = r0.copy()
    for win in range(2):
        batch = gen.make_asymspec_batch(w.recipe, 700 + V + win, B, K, V, dtype)
        a, b, t, d = _dev(batch)
        out = asv.asymspec_sci_verify(a, b, t, d, 1.0, 0.5, r_gpu)
        torch.cuda.synchronize()
        ref_a = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.0, 0.5)
        ref_s = oracle.sci_verify(batch.a, batch.t, batch.drafts, r_ref)
        st = out.req_status.cpu().numpy().astype(np.uint32)
        np.testing.assert_array_equal(st & 3, ref_a.flags & 3)
        r_new = r_gpu.cpu().numpy()
        for r in range(B):
            if not (ref_a.flags[r] & oracle.FLAGS_UNGRADED):
                assert out.accept_len[r].item() == ref_a.accept_len[r]
                np.testing.assert_array_equal(out.tokens[r].cpu().numpy(), ref_a.tokens[r])
            if not (ref_s.flags[r] & oracle.FLAGS_UNGRADED):
                assert out.sci_accept_len[r].item() == ref_s.accept_len[r]
                np.testing.assert_array_equal(out.sci_tokens[r].cpu().numpy(), ref_s.tokens[r])
                assert r_new[r] == pytest.approx(ref_s.r_hat[r], abs=1e-15)
        fin = (ref_a.flags & 1) == 0
        np.testing.assert_allclose(out.D.cpu().numpy()[fin], ref_a.D[fin], atol=tol(dtype), rtol=0)
        np.testing.assert_allclose(out.jsd.cpu().numpy()[fin], ref_s.jsd[fin], atol=tol(dtype), rtol=0)
        np.testing.assert_allclose(out.T.cpu().numpy(), ref_s.T, atol=1e-7)
        r_ref = ref_s.r_hat
