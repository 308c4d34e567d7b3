"""CUDA-graph capture of the verification calls: a call captured once (with its workspace and
outputs allocated beforehand) and replayed gives the same outputs as the same call made directly,
on the captured inputs and after new values are copied into them.  RAPID's two launches (the draw a
programmatic dependent of the verification) are captured as such; AsymSpec and E2-SCI are one
launch each.  A workspace is left zeroed by every call, so replays need no reset."""
import numpy as np
import pytest
import torch

import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def asv():
    import speculative_decoding_logit_gb300 as m
    m.build()
    return m


def _capture(call):
    """Warm up on a side stream (as torch's graph capture asks), then capture one call."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    torch.cuda.synchronize()
    return g


def _same(a, b):
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_rapid_replay_matches_direct_calls(asv):
    B, G, V = 6, 4, 8192
    b1 = gen.make_rapid_batch(11, B, G, V)
    b2 = gen.make_rapid_batch(12, B, G, V)
    z = torch.from_numpy(b1.z).cuda()
    q = torch.from_numpy(b1.q).cuda()
    d = torch.from_numpy(b1.drafts).cuda()
    ws = torch.zeros(asv.workspace_bytes(asv.ASV_MODE_RAPID, B, G, V, asv.ASV_F32), dtype=torch.uint8, device="cuda")
    out = asv.RapidOutput(torch.empty(B, dtype=torch.int32, device="cuda"),
                          torch.empty(B, G + 1, dtype=torch.int32, device="cuda"),
                          torch.empty(B, dtype=torch.int32, device="cuda"))
    call = lambda: asv.rapid_verify(z, q, d, 1.0, 10.0, 0.1, 77, out=out, workspace=ws)
    g = _capture(call)
    for batch in (b1, b2, b1):
        z.copy_(torch.from_numpy(batch.z))
        q.copy_(torch.from_numpy(batch.q))
        d.copy_(torch.from_numpy(batch.drafts))
        g.replay()
        torch.cuda.synchronize()
        got = (out.accept_len.clone(), out.tokens.clone(), out.req_status.clone())
        ref = asv.rapid_verify(z.clone(), q.clone(), d.clone(), 1.0, 10.0, 0.1, 77)
        torch.cuda.synchronize()
        _same(got, (ref.accept_len, ref.tokens, ref.req_status))
    assert not ws.any(), "the workspace is left zeroed"


def test_asymspec_replay_matches_direct_calls(asv):
    B, K, V = 8, 3, 8192
    b1 = gen.make_asymspec_batch("gumbel_zipf", 21, B, K, V, gen.BF16, processes=0)
    b2 = gen.make_asymspec_batch("gumbel_zipf", 22, B, K, V, gen.BF16, processes=0)
    todev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    a, b, t = todev(b1.a), todev(b1.b), todev(b1.t)
    d = torch.from_numpy(b1.drafts).cuda()
    ws = torch.zeros(asv.workspace_bytes(asv.ASV_MODE_ASYMSPEC, B, K, V, asv.ASV_BF16), dtype=torch.uint8, device="cuda")
    out = asv.AsymSpecOutput(torch.empty(B, dtype=torch.int32, device="cuda"),
                             torch.empty(B, K + 1, dtype=torch.int32, device="cuda"),
                             torch.empty(B, K + 1, dtype=torch.float32, device="cuda"),
                             torch.empty(B, K + 1, 3, dtype=torch.float32, device="cuda"),
                             torch.empty(B, dtype=torch.int32, device="cuda"))
    call = lambda: asv.asymspec_verify(a, b, t, d, 1.0, 0.5, out=out, workspace=ws)
    g = _capture(call)
    for batch in (b1, b2):
        for dst, src in ((a, batch.a), (b, batch.b), (t, batch.t)):
            dst.copy_(todev(src))
        d.copy_(torch.from_numpy(batch.drafts))
        g.replay()
        torch.cuda.synchronize()
        got = tuple(x.clone() for x in (out.accept_len, out.tokens, out.D, out.lse, out.req_status))
        ref = asv.asymspec_verify(a.clone(), b.clone(), t.clone(), d.clone(), 1.0, 0.5)
        torch.cuda.synchronize()
        _same(got, (ref.accept_len, ref.tokens, ref.D, ref.lse, ref.req_status))
    assert not ws.any(), "the workspace is left zeroed"


def _capture_returning(call):
    """As _capture, returning the captured call's outputs too (allocated from the graph's pool)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = call()
    torch.cuda.synchronize()
    return g, out


def test_sweep_replay_matches_direct_calls(asv):
    B, K, V = 6, 4, 4096
    b1 = gen.make_asymspec_batch("spiky", 41, B, K, V, gen.F32, identical_frac=0.3, processes=0)
    b2 = gen.make_asymspec_batch("spiky", 42, B, K, V, gen.F32, identical_frac=0.3, processes=0)
    a, b, t = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (b1.a, b1.b, b1.t))
    d = torch.from_numpy(b1.drafts).cuda()
    betas, gammas = [0.0, 1.0, 1.5, 2.0], [0.4, 0.5, 0.7, 1.0]
    ws = torch.zeros(asv.workspace_bytes(asv.ASV_MODE_SWEEP, B, K, V, asv.ASV_F32), dtype=torch.uint8, device="cuda")
    g, out = _capture_returning(lambda: asv.asymspec_verify_sweep(a, b, t, d, betas, gammas, workspace=ws))
    for batch in (b1, b2):
        for dst, src in ((a, batch.a), (b, batch.b), (t, batch.t)):
            dst.copy_(torch.from_numpy(np.ascontiguousarray(src)))
        d.copy_(torch.from_numpy(batch.drafts))
        g.replay()
        torch.cuda.synchronize()
        got = tuple(x.clone() for x in (out.accept_len, out.tokens, out.D, out.lse, out.req_status))
        ref = asv.asymspec_verify_sweep(a.clone(), b.clone(), t.clone(), d.clone(), betas, gammas)
        torch.cuda.synchronize()
        _same(got, (ref.accept_len, ref.tokens, ref.D, ref.lse, ref.req_status))
    assert not ws.any(), "the workspace is left zeroed"


def test_sci_replay_carries_the_credit_state(asv):
    """Three E2-SCI windows replayed from one capture: r_hat, updated in place on the device by each
    window, follows the same values as three direct calls."""
    B, K, V = 8, 4, 4096
    wins = [gen.make_asymspec_batch("spiky", 61 + w, B, K, V, gen.BF16, processes=0) for w in range(3)]
    todev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    dr, tg = todev(wins[0].a), todev(wins[0].t)
    d = torch.from_numpy(wins[0].drafts).cuda()
    r = torch.full((B,), 0.6, dtype=torch.float64, device="cuda")
    ws = torch.zeros(asv.workspace_bytes(asv.ASV_MODE_SCI, B, K, V, asv.ASV_BF16), dtype=torch.uint8, device="cuda")
    g, out = _capture_returning(lambda: asv.sci_verify(dr, tg, d, r, workspace=ws))
    r.fill_(0.6)  # (the warm-up call advanced it)
    r_ref = torch.full((B,), 0.6, dtype=torch.float64, device="cuda")
    for win in wins:
        dr.copy_(todev(win.a))
        tg.copy_(todev(win.t))
        d.copy_(torch.from_numpy(win.drafts))
        g.replay()
        torch.cuda.synchronize()
        got = tuple(x.clone() for x in (out.accept_len, out.tokens, out.jsd, out.T, out.req_status))
        ref = asv.sci_verify(dr.clone(), tg.clone(), d.clone(), r_ref)
        torch.cuda.synchronize()
        _same(got, (ref.accept_len, ref.tokens, ref.jsd, ref.T, ref.req_status))
        assert torch.equal(r, r_ref)
    assert not ws.any(), "the workspace is left zeroed"
