"""Helpers for the GPU parity tests: move generator batches to the device and compare the
library's outputs with the oracle's."""
import numpy as np
import torch

import gen
import oracle


def to_device(x: np.ndarray, dtype: int, device="cuda"):
    if dtype == gen.F32:
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(device)


def tol(dtype):
    # agreement bar for D and log-sum-exp: 1e-5 absolute (fp32 inputs), 2e-3 (bf16 inputs)
    return 1e-5 if dtype == gen.F32 else 2e-3


def compare_asymspec(gpu, ref: "oracle.AsymSpecResult", dtype, rows=None):
    """Returns (graded, flagged) request counts; asserts decisions/tokens bit-exact on graded
    requests and D / lse within tolerance on finite rows."""
    acc = gpu.accept_len.cpu().numpy()
    tok = gpu.tokens.cpu().numpy()
    D = gpu.D.cpu().numpy().astype(np.float64)
    lse = gpu.lse.cpu().numpy().astype(np.float64)
    st = gpu.req_status.cpu().numpy().astype(np.uint32)
    np.testing.assert_array_equal(st & 3, ref.flags & 3)
    assert not (st & 4).any(), "a bounded wait expired (ASV_REQ_TIMEOUT)"
    graded = flagged = 0
    for r in range(len(acc)):
        if ref.flags[r] & oracle.FLAGS_UNGRADED:
            flagged += 1
            continue
        graded += 1
        assert acc[r] == ref.accept_len[r], f"request {r}: accept {acc[r]} vs {ref.accept_len[r]}"
        np.testing.assert_array_equal(tok[r], ref.tokens[r], err_msg=f"request {r}")
    fin = (ref.flags & 1) == 0
    if fin.any():
        np.testing.assert_allclose(D[fin], ref.D[fin], atol=tol(dtype), rtol=0)
        np.testing.assert_allclose(lse[fin], ref.lse[fin], atol=tol(dtype), rtol=0)
    return graded, flagged
