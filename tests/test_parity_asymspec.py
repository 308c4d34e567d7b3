"""GPU parity: the CUDA AsymSpec path against the CPU oracle on the same seeded inputs.
Decisions and tokens bit-exact (requests the oracle flags as within 1e-6 of the gate are
counted, not graded); D and log-sum-exp within 1e-5 (fp32) / 2e-3 (bf16)."""
import math

import numpy as np
import pytest
import torch

import gen
import oracle
from parity_util import compare_asymspec, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def asv():
    import speculative_decoding_logit_gb300 as m
    m.build()
    assert torch.cuda.is_available()
    return m


def run(asv, batch, beta, gamma):
    a = to_device(batch.a, batch.dtype)
    b = to_device(batch.b, batch.dtype)
    t = to_device(batch.t, batch.dtype)
    d = torch.from_numpy(batch.drafts).cuda()
    out = asv.asymspec_verify(a, b, t, d, beta, gamma)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
@pytest.mark.parametrize("V", [2, 17, 1000, 1001, 4096, 32000])
def test_small_shapes(asv, dtype, V):
    batch = gen.make_asymspec_batch("spiky", 5 + V, 12, 3, V, dtype, identical_frac=0.25)
    for beta, gamma in [(1.0, 0.5), (0.0, 1.0), (2.0, 0.4)]:
        out = run(asv, batch, beta, gamma)
        ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, beta, gamma)
        graded, flagged = compare_asymspec(out, ref, dtype)
        assert graded >= 10
        ident = batch.identical
        assert np.all(out.D.cpu().numpy()[ident] == 0.0)


@pytest.mark.parametrize("K", [0, 1, 7])
def test_draft_counts(asv, K):
    batch = gen.make_asymspec_batch("gumbel_zipf", 40 + K, 9, K, 3000, gen.BF16)
    out = run(asv, batch, 1.0, 0.5)
    ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.0, 0.5)
    compare_asymspec(out, ref, gen.BF16)


def test_workspace_left_zeroed(asv):
    # Calls of growing size share one workspace; each must leave all of it zero, because a later
    # call lays its request tickets over the bytes an earlier one used for row records.
    shapes = [(9, 0, 3000), (9, 1, 3000), (12, 3, 8192), (3, 7, 32000), (20, 2, 1000)]
    need = max(asv.workspace_bytes(asv.ASV_MODE_ASYMSPEC, B, K, V, asv.ASV_BF16) for B, K, V in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for B, K, V in shapes:
        batch = gen.make_asymspec_batch("gumbel_zipf", 90 + B + K, B, K, V, gen.BF16)
        a, b, t = (to_device(x, batch.dtype) for x in (batch.a, batch.b, batch.t))
        out = asv.asymspec_verify(a, b, t, torch.from_numpy(batch.drafts).cuda(), 1.0, 0.5, workspace=ws)
        torch.cuda.synchronize()
        ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.0, 0.5)
        compare_asymspec(out, ref, gen.BF16)
        assert int(torch.count_nonzero(ws)) == 0, f"workspace not cleared after B={B} K={K} V={V}"


def test_empty_batch(asv):
    z = torch.zeros(0, 3, 100, device="cuda")
    d = torch.zeros(0, 2, dtype=torch.int32, device="cuda")
    out = asv.asymspec_verify(z, z, z, d, 1.0, 0.5)
    assert out.accept_len.numel() == 0


def test_nonfinite_and_bad_drafts(asv):
    batch = gen.make_asymspec_batch("spiky", 77, 6, 2, 500, gen.F32)
    a, b, t = batch.a.copy(), batch.b.copy(), batch.t.copy()
    d = batch.drafts.copy()
    a[1, 0, 7] = np.nan
    t[2, 2, 0] = np.inf
    b[3, 1, :] = -np.inf
    d[4, 1] = 500
    b[5, 0, 3] = -np.inf  # a single -inf is a legal logit
    out = asv.asymspec_verify(to_device(a, 0), to_device(b, 0), to_device(t, 0), torch.from_numpy(d).cuda(), 1.0, 0.5)
    torch.cuda.synchronize()
    ref = oracle.asymspec_verify(a, b, t, d, 1.0, 0.5)
    st = out.req_status.cpu().numpy()
    assert list(st) == [0, 1, 1, 1, 2, 0]
    compare_asymspec(out, ref, gen.F32)


def test_repeat_calls_reuse_workspace(asv):
    batch = gen.make_asymspec_batch("spiky", 3, 20, 2, 2048, gen.BF16)
    first = run(asv, batch, 1.0, 0.5)
    for _ in range(3):
        again = run(asv, batch, 1.0, 0.5)
        assert torch.equal(first.tokens, again.tokens) and torch.equal(first.D, again.D)


@pytest.mark.parametrize("cluster", [1, 2, 3, 8, 16])
def test_cluster_sizes_agree(asv, cluster):
    batch = gen.make_asymspec_batch("spiky", 11, 8, 2, 8192, gen.F32)
    try:
        asv.set_tuning(cluster, 256)
        out = run(asv, batch, 1.0, 0.5)
    finally:
        asv.set_tuning(0, 0)
    ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.0, 0.5)
    compare_asymspec(out, ref, gen.F32)


def test_b1_k2_v32000_f32(asv):
    w = gen.WORKLOADS["asymspec_b1_k2_v32000_f32"]
    batch = gen.make_asymspec_batch(w.recipe, w.seed, w.B, w.K, w.V, w.dtype)
    out = run(asv, batch, 1.0, 0.5)
    ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.0, 0.5)
    compare_asymspec(out, ref, w.dtype)


def test_b64_k2_v151936_bf16_full(asv):
    """The benchmarked workload, every request, both (beta, gamma) runs."""
    w = gen.WORKLOADS["asymspec_b64_k2_v151936_bf16"]
    batch = gen.make_asymspec_batch(w.recipe, w.seed, w.B, w.K, w.V, w.dtype, processes=8)
    tot_g = tot_f = 0
    for beta, gamma in w.params["runs"]:
        out = run(asv, batch, beta, gamma)
        ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, beta, gamma)
        g, f = compare_asymspec(out, ref, w.dtype)
        tot_g += g
        tot_f += f
        if beta == 0.0:
            # the degenerate run emits argmax t at the stop position
            tok = out.tokens.cpu().numpy()
            for r in range(w.B):
                n = int(out.accept_len[r])
                assert tok[r, n] == int(np.argmax(gen.widen(batch.t[r, n], w.dtype)))
    assert tot_f <= 0.05 * (tot_g + tot_f)


@pytest.mark.parametrize("src", [1, 2])
@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_delta_source_ablation(asv, src, dtype):
    """The ablation's alternative context-gain signals (delta := a, delta := t - b)."""
    batch = gen.make_asymspec_batch("spiky", 60 + src, 16, 3, 5000, dtype)
    a, b, t = (to_device(x, dtype) for x in (batch.a, batch.b, batch.t))
    d = torch.from_numpy(batch.drafts).cuda()
    for beta in (1.0, 2.0):
        out = asv.asymspec_verify(a, b, t, d, beta, 0.5, delta_source=src)
        torch.cuda.synchronize()
        ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, beta, 0.5, delta_source=src)
        compare_asymspec(out, ref, dtype)
        np.testing.assert_array_equal(out.tokens.cpu().numpy()[:, 0] >= 0, True)


@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_divergence_forms_across_their_domains(asv, dtype):
    """Rows whose per-entry log-ratio u spreads over [-7, 7]: every 16-byte vector mixes entries of
    the short narrow form (|u| <= 3), the |u| <= 4 narrow form (taken entry by entry) and the wide
    form, and in one request every entry lies in the short domain while the sums of u^2 over a
    vector exceed it (the vector test is on the largest u^2).  D agrees with the oracle far inside
    the tolerance (the fitted forms are good to ~1.6e-7 relative)."""
    B, K, V = 6, 2, 12288
    rng = np.random.default_rng(20261202 + dtype)
    a = rng.normal(0.0, 1.5, size=(B, K + 1, V))
    shift = rng.uniform(-7.0, 7.0, size=(B, K + 1, V)) * (rng.random((B, K + 1, V)) < 0.4)
    # request 4: u of every entry inside the short domain, most vectors' sums of u^2 outside it
    shift[4] = rng.uniform(-2.9, 2.9, size=(K + 1, V)) * (rng.random((K + 1, V)) < 0.9)
    b = a + shift
    t = b + rng.normal(0.0, 1.0, size=(B, K + 1, V))
    a_s, b_s, t_s = (gen.store(x, dtype) for x in (a, b, t))
    drafts = np.argmax(gen.widen(a_s, dtype)[:, :K], axis=-1).astype(np.int32)
    out = asv.asymspec_verify(to_device(a_s, dtype), to_device(b_s, dtype), to_device(t_s, dtype),
                              torch.from_numpy(drafts).cuda(), 1.0, 0.5)
    torch.cuda.synchronize()
    ref = oracle.asymspec_verify(a_s, b_s, t_s, drafts, 1.0, 0.5)
    compare_asymspec(out, ref, dtype)
    D = out.D.cpu().numpy().astype(np.float64)
    assert np.all(ref.D > 0.05)  # the rows are far from identical
    np.testing.assert_allclose(D, ref.D, rtol=2e-6, atol=0)
