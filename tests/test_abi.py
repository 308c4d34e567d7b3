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
    # tickets padded to 256 B + 16-byte row records (AsymSpec/SCI) or 32-byte (RAPID)
    assert lib.asv_workspace_bytes(0, 64, 2, 151936, 1) == 256 + 64 * 3 * 16
    # RAPID: tickets, row records (to a 256-byte boundary), one draw job per request
    assert lib.asv_workspace_bytes(1, 32, 10, 128256, 0) == 256 + 32 * 11 * 32 + 32 * 64
    assert lib.asv_workspace_bytes(0, -1, 2, 10, 0) == 0


def test_host_validation_without_gpu(lib):
    f = lib.asymspec_verify
    vp = C.c_void_p
    f.argtypes = [vp, vp, vp, C.c_int, vp, C.c_int, C.c_int, C.c_int, C.c_float, C.c_float, vp, vp, vp, vp, vp, vp,
                  C.c_size_t, vp]
    P = 1 << 20  # a non-null, 256-aligned stand-in address (never dereferenced: calls fail first)

    def call(B=2, K=2, V=64, dt=0, beta=1.0, gamma=0.5, a=P, ws=P, wsb=1 << 20, d=P):
        return f(a, P, P, dt, d, B, K, V, beta, gamma, P, P, P, P, P, ws, wsb, None)

    assert call(B=-1) == 2
    assert call(K=-1) == 2
    assert call(V=1) == 2
    assert call(dt=5) == 4
    assert call(B=0) == 0                      # empty batch is a no-op
    assert call(a=None) == 1
    assert call(d=None) == 1
    assert call(ws=None) == 6
    assert call(a=P + 2) == 3                  # fp32 input not 4-byte aligned
    assert call(gamma=0.0) == 5
    assert call(gamma=float("nan")) == 5
    assert call(beta=float("inf")) == 5
    assert call(wsb=16) == 6                   # workspace too small


def test_tuning_override_validation(lib):
    assert lib.asv_set_tuning(17, 0) == 5
    assert lib.asv_set_tuning(4, 100) == 5
    assert lib.asv_set_tuning(4, 256) == 0
    assert lib.asv_set_tuning(0, 0) == 0
