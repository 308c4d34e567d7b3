"""GPU parity for the E2-SCI window: JSD within tolerance, accept lengths and tokens
bit-exact (requests within 1e-6 of the threshold counted, not graded), credit state
carried across windows identically."""
import numpy as np
import pytest
import torch

import gen
import oracle
from parity_util import to_device, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def asv():
    import speculative_decoding_logit_gb300 as m
    m.build()
    return m


def _window(asv, batch, r_hat, params=None):
    p = params or asv.SciParams()
    r = torch.from_numpy(np.array(r_hat, np.float64)).cuda()
    out = asv.sci_verify(to_device(batch.a, batch.dtype), to_device(batch.t, batch.dtype),
                         torch.from_numpy(batch.drafts).cuda(), r, p)
    torch.cuda.synchronize()
    op = oracle.SciParams(p.T_base, p.alpha_omega, p.tau_credit, p.T_min, p.T_max, p.ewma_beta)
    ref = oracle.sci_verify(batch.a, batch.t, batch.drafts, r_hat, op)
    return out, r.cpu().numpy(), ref


def _compare(out, r_new, ref, dtype):
    st = out.req_status.cpu().numpy().astype(np.uint32)
    np.testing.assert_array_equal(st & 3, ref.flags & 3)
    assert not (st & 4).any(), "a bounded wait expired (ASV_REQ_TIMEOUT)"
    acc = out.accept_len.cpu().numpy()
    tok = out.tokens.cpu().numpy()
    graded = 0
    for r in range(len(acc)):
        if ref.flags[r] & oracle.FLAGS_UNGRADED:
            continue
        graded += 1
        assert acc[r] == ref.accept_len[r]
        np.testing.assert_array_equal(tok[r], ref.tokens[r])
        assert r_new[r] == pytest.approx(ref.r_hat[r], abs=1e-15)
    fin = (ref.flags & 1) == 0
    np.testing.assert_allclose(out.jsd.cpu().numpy()[fin], ref.jsd[fin], atol=tol(dtype), rtol=0)
    np.testing.assert_allclose(out.T.cpu().numpy(), ref.T, atol=1e-7)
    return graded


@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
@pytest.mark.parametrize("V", [33, 2048, 151936])
def test_window_shapes(asv, dtype, V):
    B = 16 if V < 100000 else 4
    batch = gen.make_asymspec_batch("spiky", 900 + V, B, 8, V, dtype)
    rng = np.random.default_rng(V)
    out, r_new, ref = _window(asv, batch, rng.uniform(0, 1, B))
    assert _compare(out, r_new, ref, dtype) >= B - 2


def test_clamps_bind(asv):
    batch = gen.make_asymspec_batch("spiky", 5, 8, 4, 1000, gen.BF16)
    p = asv.SciParams(alpha_omega=2.0)
    out, r_new, ref = _window(asv, batch, np.linspace(0, 1, 8), p)
    T = out.T.cpu().numpy()
    assert T.min() == pytest.approx(0.1) and T.max() == pytest.approx(0.6)
    _compare(out, r_new, ref, gen.BF16)


def test_stabilised_windows(asv):
    """Six windows with hysteresis, a refresh interval of 2 and a fallback, state on the device."""
    B, K, V = 24, 4, 4096
    stab = asv.SciStabilisers(hysteresis=0.01, min_refresh=2, fallback_acc=0.5, fallback_T=0.12)
    ostab = oracle.SciStabilisers(0.01, 2, 0.5, 0.12)
    p = asv.SciParams(alpha_omega=0.5)
    op = oracle.SciParams(p.T_base, p.alpha_omega, p.tau_credit, p.T_min, p.T_max, p.ewma_beta)
    state = asv.sci_state_new(B)
    ostate = oracle.sci_state(B)
    rng = np.random.default_rng(31)
    r_ref = rng.uniform(0.2, 1.0, B)
    r_gpu = torch.from_numpy(r_ref.copy()).cuda()
    applied_fallback = 0
    for win in range(6):
        batch = gen.make_asymspec_batch("spiky", 4000 + win, B, K, V, gen.F32)
        out = asv.sci_verify(to_device(batch.a, batch.dtype), to_device(batch.t, batch.dtype),
                             torch.from_numpy(batch.drafts).cuda(), r_gpu, p, stabilisers=stab, state=state)
        torch.cuda.synchronize()
        ref = oracle.sci_verify(batch.a, batch.t, batch.drafts, r_ref, op, stab=ostab, state=ostate)
        _compare(out, r_gpu.cpu().numpy(), ref, gen.F32)
        T_app, age, flags = asv.sci_state_decode(state)
        for r in range(B):
            if ref.flags[r] & oracle.FLAGS_UNGRADED:
                continue
            assert T_app[r].item() == pytest.approx(ostate[r].T_applied, abs=1e-15)
            assert age[r].item() == ostate[r].age and flags[r].item() == ostate[r].flags
        applied_fallback += int(np.isclose(ref.T, 0.12).sum())
        r_ref = ref.r_hat
    assert applied_fallback > 0  # the fallback path ran


@pytest.mark.parametrize("dtype,V", [(gen.F32, 2048), (gen.BF16, 8192), (gen.F32, 1001)])
def test_prehit_equals_full_window(asv, dtype, V):
    """First-token pre-hit: a window whose first draft fails is dropped without reading its later
    rows; for finite inputs the decisions, tokens, thresholds and credit equal the full window's."""
    B, K = 32, 6
    rng = np.random.default_rng(V)
    batch = gen.make_asymspec_batch("spiky", 1200 + V, B, K, V, dtype)
    r0 = rng.uniform(0.0, 1.0, B)
    p = asv.SciParams(alpha_omega=1.0)   # thresholds spread over [0.1, 0.6]
    op = oracle.SciParams(p.T_base, p.alpha_omega, p.tau_credit, p.T_min, p.T_max, p.ewma_beta)
    r_gpu = torch.from_numpy(r0.copy()).cuda()
    out = asv.sci_verify(to_device(batch.a, batch.dtype), to_device(batch.t, batch.dtype),
                         torch.from_numpy(batch.drafts).cuda(), r_gpu, p, prehit=True)
    torch.cuda.synchronize()
    ref = oracle.sci_verify(batch.a, batch.t, batch.drafts, r0, op)
    st = out.req_status.cpu().numpy().astype(np.uint32)
    np.testing.assert_array_equal(st & 3, ref.flags & 3)
    acc = out.accept_len.cpu().numpy()
    tok = out.tokens.cpu().numpy()
    jsd = out.jsd.cpu().numpy()
    r_new = r_gpu.cpu().numpy()
    dropped = graded = 0
    for r in range(B):
        if ref.flags[r] & oracle.FLAGS_UNGRADED:
            continue
        graded += 1
        assert acc[r] == ref.accept_len[r]
        np.testing.assert_array_equal(tok[r], ref.tokens[r])
        assert r_new[r] == pytest.approx(ref.r_hat[r], abs=1e-15)
        cols = 1 if ref.accept_len[r] == 0 else K + 1   # a dropped window has only row 0's J
        dropped += int(ref.accept_len[r] == 0)
        np.testing.assert_allclose(jsd[r, :cols], ref.jsd[r, :cols], atol=tol(dtype), rtol=0)
    np.testing.assert_allclose(out.T.cpu().numpy(), ref.T, atol=1e-7)
    assert graded >= B - 4 and dropped >= 3
    # the workspace is left zeroed (the drop flags are cleared)
    for buf in asv._binding._ws_cache.values():
        assert int(torch.count_nonzero(buf)) == 0
