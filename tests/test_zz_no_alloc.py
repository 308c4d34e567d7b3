"""asymspec_verify_static, the entry point for callers that cannot allocate device memory
(for instance a plugin handed only its input and output buffers by a serving framework, or
code that must not allocate once running): it keeps its scratch in a library-owned static
device array.  Checked through the C ABI against asymspec_verify (caller workspace) on two
calls in a row, and for the size limit.  This file is collected last on purpose."""
import ctypes as C
import os
import re

import numpy as np
import pytest
import torch

import gen

pytestmark = pytest.mark.gpu


def _static_scratch_bytes():
    """ASV_STATIC_SCRATCH_BYTES as include/asv.h defines it (read from the header, so the limit a
    test relies on cannot drift from the library's)."""
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "asv.h")
    m = re.search(r"#define\s+ASV_STATIC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", open(hdr).read())
    assert m, "ASV_STATIC_SCRATCH_BYTES not found in asv.h"
    return int(m.group(1)) << int(m.group(2))


def _to_dev(x, dtype):
    if dtype == gen.F32:
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def _static_call(lib, a, b, t, d, dtype, B, K, V, beta, gamma):
    f = lib.asymspec_verify_static
    vp = C.c_void_p
    f.argtypes = [vp, vp, vp, C.c_int, vp, C.c_int, C.c_int, C.c_int, C.c_float, C.c_float, vp, vp, vp, vp, vp, vp]
    f.restype = C.c_int
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    tok = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
    D = torch.full((B, K + 1), -1.0, dtype=torch.float32, device="cuda")
    lse = torch.full((B, K + 1, 3), -1.0, dtype=torch.float32, device="cuda")
    st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = f(a.data_ptr(), b.data_ptr(), t.data_ptr(), dtype, d.data_ptr(), B, K, V, beta, gamma, acc.data_ptr(),
           tok.data_ptr(), D.data_ptr(), lse.data_ptr(), st.data_ptr(), stream)
    torch.cuda.synchronize()
    return rc, acc, tok, D, lse, st


def test_static_scratch_matches_workspace_entry_point():
    import speculative_decoding_logit_gb300 as asv
    asv.build()
    lib = asv.library()
    cases = [(gen.BF16, "gumbel_zipf", 12, 3, 6000, 1.0, 0.5, 401),
             (gen.F32, "spiky", 9, 2, 4099, 0.0, 1.0, 402)]   # second call: other shape, unaligned rows
    for dtype, recipe, B, K, V, beta, gamma, seed in cases:
        batch = gen.make_asymspec_batch(recipe, seed, B, K, V, dtype)
        a, b, t = (_to_dev(x, dtype) for x in (batch.a, batch.b, batch.t))
        d = torch.from_numpy(batch.drafts).cuda()
        ref = asv.asymspec_verify(a, b, t, d, beta, gamma)
        torch.cuda.synchronize()
        rc, acc, tok, D, lse, st = _static_call(lib, a, b, t, d, dtype, B, K, V, beta, gamma)
        assert rc == 0
        assert torch.equal(acc, ref.accept_len) and torch.equal(tok, ref.tokens)
        assert torch.equal(st, ref.req_status)
        tol = 1e-5 if dtype == gen.F32 else 2e-3
        assert torch.allclose(D, ref.D, atol=tol, rtol=0) and torch.allclose(lse, ref.lse, atol=tol, rtol=0)


def test_static_scratch_rejects_batches_beyond_its_size():
    import speculative_decoding_logit_gb300 as asv
    asv.build()
    lib = asv.library()
    K, V = 8, 1000
    B = 200000   # about 2 million rows: a workspace far beyond the static scratch
    need = lib.asv_workspace_bytes(0, B, K, V, 1)
    limit = _static_scratch_bytes()
    # Every pointer is NULL: the size check must reject the batch first (ASV_ERR_WORKSPACE); if it
    # ever let the batch through, the argument checks that follow it stop the call at ASV_ERR_NULL
    # on the host.  Either way nothing reaches the GPU.
    f = lib.asymspec_verify_static
    vp = C.c_void_p
    f.argtypes = [vp, vp, vp, C.c_int, vp, C.c_int, C.c_int, C.c_int, C.c_float, C.c_float, vp, vp, vp, vp, vp, vp]
    f.restype = C.c_int
    assert f(None, None, None, 1, None, B, K, V, 1.0, 0.5, None, None, None, None, None, None) == 6
    # Within the limit, the same all-NULL call ends at the argument checks, before any CUDA call.
    assert f(None, None, None, 1, None, 4, K, V, 1.0, 0.5, None, None, None, None, None, None) == 1
