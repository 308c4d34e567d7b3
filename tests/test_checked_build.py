"""Memory-safety checks without a sanitizer: the bounds-checked library (-DASV_CHECKED: every global
and shared-memory index the kernels form is tested against its buffer; a failed test is counted in
the workspace's check log and the access is skipped, nothing traps), driven through the C ABI with
a canary region after every output buffer and after the workspace.  Each call must leave its check
log at zero, every canary intact, the rest of the workspace zero, and its decisions equal to the
oracle's.  The shapes cover tiny and odd vocabularies (V = 2, 17, 1001, 4099), odd draft counts,
cluster sizes 1-16 and both AsymSpec kernels ("AsymSpec: Context-Asymmetric Speculative Decoding
for Agentic LLMs", sec. 4.1-4.2; "E2-SCI: Elastic Edge-Cloud Speculative Decoding via Credit
Inertia", Key design 3; "RAPID: Long-Context Inference with Retrieval-Augmented Speculative
Decoding", Key designs 2-4)."""
import ctypes as C
import os

import numpy as np
import pytest
import torch

import gen
import oracle
from parity_util import to_device

CANARY = 0x5A5A5A5A
GUARD = 64  # canary words after each buffer


@pytest.fixture(scope="module")
def clib():
    from speculative_decoding_logit_gb300 import _binding, nvcc_build
    path = nvcc_build.build_checked()
    lib = C.CDLL(path)
    _binding._declare(lib)
    return lib


def test_checked_library_exports_the_abi(clib):
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "asv.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    for name in set(re.findall(r"^(?:asv_status|size_t|const char\*|int)\s+(\w+)\s*\(", hdr, flags=re.M)):
        assert hasattr(clib, name), name


class Guarded:
    """A device buffer of `n` elements followed by GUARD canary words."""

    def __init__(self, n, dtype):
        words = (n * torch.tensor([], dtype=dtype).element_size() + 3) // 4
        self.raw = torch.full((words + GUARD,), CANARY, dtype=torch.int32, device="cuda")
        self.t = self.raw[:words].view(dtype)[:n] if n else self.raw[:0].view(dtype)
        self.words = words

    def ptr(self):
        return self.raw.data_ptr()

    def intact(self):
        return bool(torch.all(self.raw[self.words:] == CANARY))


class Workspace:
    def __init__(self, nbytes):
        self.n = nbytes
        self.raw = torch.zeros(nbytes + 4 * GUARD, dtype=torch.uint8, device="cuda")
        self.raw[nbytes:].view(torch.int32).fill_(CANARY)

    def ptr(self):
        return self.raw.data_ptr()

    def check(self):
        """(violations counted, line of the first), with the canary and the zero-fill verified."""
        assert bool(torch.all(self.raw[self.n:].view(torch.int32) == CANARY)), "workspace canary overwritten"
        log = self.raw[self.n - 256:self.n].view(torch.int32).cpu().numpy()
        body = self.raw[:self.n - 256]
        count, line = int(log[0]), int(log[1])
        if count == 0:
            assert int(torch.count_nonzero(body)) == 0, "workspace not left zeroed"
        return count, line


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _asym(clib, batch, beta, gamma, cluster, kernel):
    B, R1, V = batch.a.shape
    K = R1 - 1
    dt = batch.dtype
    a, b, t = (to_device(x, dt) for x in (batch.a, batch.b, batch.t))
    d = torch.from_numpy(np.ascontiguousarray(batch.drafts)).cuda()
    assert clib.asv_set_tuning(cluster, 0) == 0 and clib.asv_set_kernel(kernel) == 0
    try:
        acc, tok, st = Guarded(B, torch.int32), Guarded(B * R1, torch.int32), Guarded(B, torch.int32)
        D, lse = Guarded(B * R1, torch.float32), Guarded(B * R1 * 3, torch.float32)
        ws = Workspace(clib.asv_workspace_bytes(0, B, K, V, dt))
        rc = clib.asymspec_verify(a.data_ptr(), b.data_ptr(), t.data_ptr(), dt, d.data_ptr(), B, K, V, beta, gamma,
                                  acc.ptr(), tok.ptr(), D.ptr(), lse.ptr(), st.ptr(), ws.ptr(), ws.n, _stream())
        torch.cuda.synchronize()
    finally:
        clib.asv_set_tuning(0, 0)
        clib.asv_set_kernel(0)
    assert rc == 0
    count, line = ws.check()
    assert count == 0, f"{count} index checks failed (first at line {line})"
    for g in (acc, tok, st, D, lse):
        assert g.intact(), "an output canary was overwritten"
    ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, beta, gamma)
    ok = (ref.flags & oracle.FLAGS_UNGRADED) == 0
    np.testing.assert_array_equal(st.t.cpu().numpy() & 3, ref.flags & 3)
    np.testing.assert_array_equal(acc.t.cpu().numpy()[ok], ref.accept_len[ok])
    np.testing.assert_array_equal(tok.t.view(B, R1).cpu().numpy()[ok], ref.tokens[ok])


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
@pytest.mark.parametrize("V", [2, 17, 1001, 4099])
def test_asymspec_checked_every_cluster_size(clib, dtype, V):
    for K in (1, 3, 7):
        batch = gen.make_asymspec_batch("spiky", 70 + V + K, 3, K, V, dtype, identical_frac=0.3)
        for cluster in range(1, 17):
            if cluster > 1 and V < 1024:
                continue  # (slices of a few entries: every size from 1 to 16 is run at V = 1001 and 4099)
            _asym(clib, batch, 1.0, 0.5, cluster, 1)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,V", [(gen.F32, 4096), (gen.BF16, 8200), (gen.BF16, 151936), (gen.F32, 32000)])
def test_asymspec_checked_staged_kernel(clib, dtype, V):
    for K in (1, 3):
        batch = gen.make_asymspec_batch("gumbel_zipf", 90 + V + K, 5, K, V, dtype)
        _asym(clib, batch, 1.5, 0.5, 0, 2)


@pytest.mark.gpu
@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("dtype,V", [(gen.F32, 1001), (gen.BF16, 4096), (gen.BF16, 151936)])
def test_sci_sweep_fused_checked(clib, kernel, dtype, V):
    from speculative_decoding_logit_gb300 import _binding
    B, K = 4, 3
    batch = gen.make_asymspec_batch("spiky", 40 + V, B, K, V, dtype)
    R1 = K + 1
    a, b, t = (to_device(x, dtype) for x in (batch.a, batch.b, batch.t))
    d = torch.from_numpy(batch.drafts).cuda()
    sp = oracle.SciParams()
    pc = _binding._SciParamsC(sp.T_base, sp.alpha_omega, sp.tau_credit, sp.T_min, sp.T_max, sp.ewma_beta)
    clib.asv_set_kernel(kernel)
    try:
        # E2-SCI window
        r = Guarded(B, torch.float64)
        r.t.fill_(0.6)
        acc, tok, jsd, T, st = (Guarded(B, torch.int32), Guarded(B * R1, torch.int32), Guarded(B * R1, torch.float32),
                                Guarded(B, torch.float32), Guarded(B, torch.int32))
        ws = Workspace(clib.asv_workspace_bytes(2, B, K, V, dtype))
        assert clib.sci_verify(a.data_ptr(), t.data_ptr(), dtype, d.data_ptr(), B, K, V, C.byref(pc), r.ptr(),
                               acc.ptr(), tok.ptr(), jsd.ptr(), T.ptr(), st.ptr(), ws.ptr(), ws.n, _stream()) == 0
        torch.cuda.synchronize()
        assert ws.check()[0] == 0 and all(g.intact() for g in (r, acc, tok, jsd, T, st))
        ref = oracle.sci_verify(batch.a, batch.t, batch.drafts, np.full(B, 0.6))
        ok = (ref.flags & oracle.FLAGS_UNGRADED) == 0
        np.testing.assert_array_equal(tok.t.view(B, R1).cpu().numpy()[ok], ref.tokens[ok])
        # the all-(beta, gamma) sweep from one read
        betas = (C.c_float * 2)(0.0, 1.5)
        gammas = (C.c_float * 3)(0.4, 0.5, 1.0)
        acc, tok, D, st = (Guarded(3 * B, torch.int32), Guarded(2 * 3 * B * R1, torch.int32),
                           Guarded(B * R1, torch.float32), Guarded(B, torch.int32))
        ws = Workspace(clib.asv_workspace_bytes(3, B, K, V, dtype))
        assert clib.asymspec_verify_sweep(a.data_ptr(), b.data_ptr(), t.data_ptr(), dtype, d.data_ptr(), B, K, V,
                                          betas, 2, gammas, 3, acc.ptr(), tok.ptr(), D.ptr(), None, st.ptr(),
                                          ws.ptr(), ws.n, _stream()) == 0
        torch.cuda.synchronize()
        assert ws.check()[0] == 0 and all(g.intact() for g in (acc, tok, D, st))
        for i, be in enumerate((0.0, 1.5)):
            for j, ga in enumerate((0.4, 0.5, 1.0)):
                ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, be, ga)
                ok = (ref.flags & oracle.FLAGS_UNGRADED) == 0
                got = tok.t.view(2, 3, B, R1).cpu().numpy()[i, j]
                np.testing.assert_array_equal(got[ok], ref.tokens[ok])
        # AsymSpec fused with E2-SCI
        r = Guarded(B, torch.float64)
        r.t.fill_(0.6)
        outs = (Guarded(B, torch.int32), Guarded(B * R1, torch.int32), Guarded(B * R1, torch.float32),
                Guarded(B * R1 * 3, torch.float32), Guarded(B, torch.int32), Guarded(B * R1, torch.int32),
                Guarded(B * R1, torch.float32), Guarded(B, torch.float32), Guarded(B, torch.int32))
        ws = Workspace(clib.asv_workspace_bytes(4, B, K, V, dtype))
        assert clib.asymspec_sci_verify(a.data_ptr(), b.data_ptr(), t.data_ptr(), dtype, d.data_ptr(), B, K, V, 1.0,
                                        0.5, C.byref(pc), r.ptr(), *[g.ptr() for g in outs], ws.ptr(), ws.n,
                                        _stream()) == 0
        torch.cuda.synchronize()
        assert ws.check()[0] == 0 and r.intact() and all(g.intact() for g in outs)
        ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.0, 0.5)
        ok = (ref.flags & oracle.FLAGS_UNGRADED) == 0
        np.testing.assert_array_equal(outs[1].t.view(B, R1).cpu().numpy()[ok], ref.tokens[ok])
    finally:
        clib.asv_set_kernel(0)


@pytest.mark.gpu
@pytest.mark.parametrize("V", [2, 17, 1001, 4099, 4096])
def test_rapid_checked_every_cluster_size(clib, V):
    for G in (1, 3, 5):
        batch = gen.make_rapid_batch(300 + V + G, 3, G, V)
        z = torch.from_numpy(batch.z).cuda()
        q = torch.from_numpy(batch.q).cuda()
        d = torch.from_numpy(batch.drafts).cuda()
        R1 = G + 1
        for cluster in range(1, 17):
            if cluster > 1 and V < 1024:
                continue
            assert clib.asv_set_tuning(cluster, 0) == 0
            try:
                acc, tok, st = Guarded(3, torch.int32), Guarded(3 * R1, torch.int32), Guarded(3, torch.int32)
                ws = Workspace(clib.asv_workspace_bytes(1, 3, G, V, 0))
                rc = clib.rapid_verify(z.data_ptr(), q.data_ptr(), d.data_ptr(), 3, G, V, 1.0, 10.0, 0.1, 1234, 0,
                                       acc.ptr(), tok.ptr(), st.ptr(), ws.ptr(), ws.n, _stream())
                torch.cuda.synchronize()
            finally:
                clib.asv_set_tuning(0, 0)
            assert rc == 0
            count, line = ws.check()
            assert count == 0, f"{count} index checks failed (first at line {line})"
            assert acc.intact() and tok.intact() and st.intact()
            ref = oracle.rapid_verify(batch.z, batch.q, batch.drafts, 1.0, 10.0, 0.1, 1234)
            ok = (ref.flags & oracle.FLAGS_UNGRADED) == 0
            np.testing.assert_array_equal(acc.t.cpu().numpy()[ok], ref.accept_len[ok])
            np.testing.assert_array_equal(tok.t.view(3, R1).cpu().numpy()[ok], ref.tokens[ok])
