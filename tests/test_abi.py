"""The C ABI library builds, loads without a GPU, exports every entry point that
include/asv.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "asv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^(?:asv_status|size_t|const char\*|int)\s+(\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import speculative_decoding_logit_gb300 as asv
    asv.build()
    return asv.library()


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("asymspec_verify", "rapid_verify", "sci_verify", "asv_workspace_bytes", "asymspec_verify_host"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_status_strings_and_workspace_sizes(lib):
    for s in range(8):
        assert lib.asv_status_string(s).startswith(b"ASV_")
    # Rows that are not whole 16-byte vectors (V = 1001 bf16) take the cluster kernel: tickets padded
    # to 256 B + 16-byte row records (AsymSpec/SCI) or 32-byte (RAPID).
    assert lib.asv_workspace_bytes(0, 64, 2, 1001, 1) == 256 + 64 * 3 * 16
    # With the staged kernel selected, aligned rows add its exchange area: two counters per row
    # (256-byte padded), the abort flag (256 B) and 128 + 64 bytes of partials per unit; V = 151936
    # bf16 (three inputs in pass A, two in pass B) is 20 units of 7600 entries per row.
    assert lib.asv_workspace_bytes(0, 64, 2, 151936, 1) == 256 + 64 * 3 * 16   # cluster kernel (default)
    rows, units = 64 * 3, 64 * 3 * 20
    assert lib.asv_set_kernel(2) == 0
    try:
        assert lib.asv_workspace_bytes(0, 64, 2, 151936, 1) == 3328 + 1536 + 256 + units * 192
        assert rows * 8 == 1536
    finally:
        lib.asv_set_kernel(0)
    # RAPID: tickets, row records (to a 256-byte boundary), one draw job per request
    assert lib.asv_workspace_bytes(1, 32, 10, 128256, 0) == 256 + 32 * 11 * 32 + 32 * 64
    assert lib.asv_workspace_bytes(0, -1, 2, 10, 0) == 0


def test_host_validation_without_gpu(lib):
    """Each case leaves every pointer NULL except the one it checks, so a regression in a check
    ends at ASV_ERR_NULL on the host: no case can reach a launch."""
    f = lib.asymspec_verify
    vp = C.c_void_p
    f.argtypes = [vp, vp, vp, C.c_int, vp, C.c_int, C.c_int, C.c_int, C.c_float, C.c_float, vp, vp, vp, vp, vp, vp,
                  C.c_size_t, vp]
    host = (C.c_uint32 * 16)()   # a real (host) allocation: misaligned addresses are taken inside it
    base = C.addressof(host)
    assert base % 4 == 0

    def call(B=2, K=2, V=64, dt=0, beta=1.0, gamma=0.5, a=None):
        return f(a, None, None, dt, None, B, K, V, beta, gamma, None, None, None, None, None, None, 1 << 20, None)

    assert call(B=-1) == 2
    assert call(K=-1) == 2
    assert call(V=1) == 2
    assert call(B=1 << 30, K=7) == 2           # B * (K + 1) beyond the launch grid
    assert call(dt=5) == 4
    assert call(B=0) == 0                      # empty batch is a no-op
    assert call(gamma=0.0) == 5
    assert call(gamma=float("nan")) == 5
    assert call(beta=float("inf")) == 5
    assert call(a=base + 2) == 3               # fp32 input not 4-byte aligned (checked before NULLs)
    assert call(a=base + 2, dt=1) == 1         # 2-byte aligned is enough for bf16: then the NULLs
    assert call() == 1                         # required pointers missing


def _sized_workspace_bytes(lib):
    return lib.asv_workspace_bytes(0, 2, 2, 64, 0)


@pytest.mark.gpu
def test_workspace_checks_with_real_buffers(lib):
    """Workspace errors need every other argument valid: real device buffers of a B=2, K=2, V=64
    fp32 batch, then a workspace that is missing, too small, misaligned, and finally sufficient."""
    import torch
    vp = C.c_void_p
    f = lib.asymspec_verify
    f.argtypes = [vp, vp, vp, C.c_int, vp, C.c_int, C.c_int, C.c_int, C.c_float, C.c_float, vp, vp, vp, vp, vp, vp,
                  C.c_size_t, vp]
    B, K, V = 2, 2, 64
    g = torch.Generator().manual_seed(5)
    a, b, t = (torch.randn(B, K + 1, V, generator=g).cuda() for _ in range(3))
    d = torch.zeros(B, K, dtype=torch.int32, device="cuda")
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    tok = torch.empty(B, K + 1, dtype=torch.int32, device="cuda")
    D = torch.empty(B, K + 1, device="cuda")
    st = torch.empty(B, dtype=torch.int32, device="cuda")
    need = _sized_workspace_bytes(lib)
    ws = torch.zeros(need + 512, dtype=torch.uint8, device="cuda")
    sh = torch.cuda.current_stream().cuda_stream

    def call(w, nbytes):
        return f(a.data_ptr(), b.data_ptr(), t.data_ptr(), 0, d.data_ptr(), B, K, V, 1.0, 0.5, acc.data_ptr(),
                 tok.data_ptr(), D.data_ptr(), None, st.data_ptr(), w, nbytes, sh)

    assert call(None, need) == 6
    assert call(ws.data_ptr(), 16) == 6
    assert call(ws.data_ptr() + 16, need) == 3      # workspace not 256-byte aligned
    assert call(ws.data_ptr(), need) == 0
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(ws)) == 0


def test_kernel_selection_validation(lib):
    assert lib.asv_set_kernel(3) == 5
    assert lib.asv_set_kernel(-1) == 5
    for k in (2, 1, 0):
        assert lib.asv_set_kernel(k) == 0


def test_tuning_override_validation(lib):
    assert lib.asv_set_tuning(17, 0) == 5
    assert lib.asv_set_tuning(4, 100) == 5
    assert lib.asv_set_tuning(4, 256) == 0
    assert lib.asv_set_tuning(0, 0) == 0
