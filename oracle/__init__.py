"""CPU oracle for the logit-space verification step -- TEST INFRASTRUCTURE.

A plain double-precision C implementation (``asv_oracle.c``) of what the
verification step computes, wrapped with ctypes.  Only the tests, the
package's smoke check and the benchmark's CPU-baseline / reference leg may
import this module; the product path never does.  It shares no code with the
CUDA library.

Readings of the pages, pins and tolerances are documented in ``asv_oracle.c``
and in the design notes.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "asv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

F32 = 0
BF16 = 1

FLAG_NONFINITE = 1
FLAG_BAD_DRAFT = 2
FLAG_NEAR_MARGIN = 4
FLAG_NEAR_TAIL = 8
FLAG_NEAR_RACE = 16
FLAG_NEAR_TIE = 32
FLAGS_UNGRADED = FLAG_NEAR_MARGIN | FLAG_NEAR_TAIL | FLAG_NEAR_RACE | FLAG_NEAR_TIE


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _declare(_lib)
    return _lib


_vp = C.c_void_p
_i32p = C.POINTER(C.c_int32)
_u32p = C.POINTER(C.c_uint32)
_f64p = C.POINTER(C.c_double)
_f32p = C.POINTER(C.c_float)


def _declare(L):
    L.oracle_lse.argtypes = [_vp, C.c_int, C.c_size_t, C.c_int, C.c_double]
    L.oracle_lse.restype = C.c_double
    L.oracle_jsd.argtypes = [_vp, _vp, C.c_int, C.c_size_t, C.c_size_t, C.c_int]
    L.oracle_jsd.restype = C.c_double
    L.oracle_fused_argmax_exact.argtypes = [_vp, _vp, _vp, C.c_int, C.c_size_t, C.c_int, C.c_double, C.c_int,
                                            C.POINTER(C.c_int)]
    L.oracle_fused_argmax_exact.restype = C.c_int
    L.oracle_fused_argmax_fp32.argtypes = [_vp, _vp, _vp, C.c_int, C.c_size_t, C.c_int, C.c_float, C.c_int]
    L.oracle_fused_argmax_fp32.restype = C.c_int
    L.oracle_asymspec_verify.argtypes = [_vp, _vp, _vp, C.c_int, _i32p, C.c_int, C.c_int, C.c_int, C.c_float,
                                         C.c_float, _i32p, _i32p, _f64p, _f64p, _f64p, _i32p, _i32p, _u32p]
    L.oracle_asymspec_verify.restype = None
    L.oracle_asymspec_verify_src.argtypes = [_vp, _vp, _vp, C.c_int, _i32p, C.c_int, C.c_int, C.c_int, C.c_float,
                                             C.c_float, C.c_int, _i32p, _i32p, _f64p, _f64p, _f64p, _i32p, _i32p,
                                             _u32p]
    L.oracle_asymspec_verify_src.restype = None
    L.oracle_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
    L.oracle_philox4x32_10.restype = None
    L.oracle_uniform_from_word.argtypes = [C.c_uint32]
    L.oracle_uniform_from_word.restype = C.c_double
    L.oracle_rapid_uniform.argtypes = [C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint32]
    L.oracle_rapid_uniform.restype = C.c_double
    L.oracle_rapid_row.argtypes = [_f32p, _f32p, C.c_int, C.c_double, C.c_double, C.c_double, _f64p, _f64p,
                                   _f64p, _f64p, C.POINTER(C.c_int)]
    L.oracle_rapid_row.restype = C.c_int
    L.oracle_race.argtypes = [_f64p, C.c_int, C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint32,
                              C.POINTER(C.c_int)]
    L.oracle_race.restype = C.c_int
    L.oracle_rapid_verify.argtypes = [_f32p, _f32p, _i32p, C.c_int, C.c_int, C.c_int, C.c_double, C.c_double,
                                      C.c_double, C.c_uint64, C.c_uint32, _i32p, _i32p, _u32p]
    L.oracle_rapid_verify.restype = None
    L.oracle_sci_threshold.argtypes = [C.c_double] * 6
    L.oracle_sci_threshold.restype = C.c_double
    L.oracle_sci_ewma.argtypes = [C.c_double] * 3
    L.oracle_sci_ewma.restype = C.c_double
    L.oracle_sci_verify.argtypes = [_vp, _vp, C.c_int, _i32p, C.c_int, C.c_int, C.c_int] + [C.c_double] * 6 + \
        [_f64p, _i32p, _i32p, _f64p, _f64p, _u32p]
    L.oracle_sci_verify.restype = None
    L.oracle_rapid_row_mode.argtypes = [_f32p, _f32p, C.c_int, C.c_double, C.c_double, C.c_double, C.c_int, _f64p,
                                        _f64p, _f64p, _f64p, C.POINTER(C.c_int)]
    L.oracle_rapid_row_mode.restype = C.c_int
    L.oracle_rapid_verify_mode.argtypes = [_f32p, _f32p, _i32p, C.c_int, C.c_int, C.c_int, C.c_double, C.c_double,
                                           C.c_double, C.c_int, C.c_uint64, C.c_uint32, _i32p, _i32p, _u32p]
    L.oracle_rapid_verify_mode.restype = None
    L.oracle_sci_stab_threshold.argtypes = [C.POINTER(SciStateC), C.c_double, C.c_double, C.c_int, C.c_double,
                                            C.POINTER(C.c_int32)]
    L.oracle_sci_stab_threshold.restype = C.c_double
    L.oracle_sci_verify_stab.argtypes = [_vp, _vp, C.c_int, _i32p, C.c_int, C.c_int, C.c_int] + \
        [C.c_double] * 7 + [C.c_int, C.c_double, C.c_double, C.POINTER(SciStateC), _f64p, _i32p, _i32p, _f64p,
                            _f64p, _u32p]
    L.oracle_sci_verify_stab.restype = None


def _p(a, ct):
    return a.ctypes.data_as(C.POINTER(ct))


def _elem_dtype(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return F32
    if x.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle inputs are float32 or uint16 (bf16 bits), got {x.dtype}")


def _c(x):
    return np.ascontiguousarray(x)


# ------------------------------------------------------------------ row helpers

def lse(x: np.ndarray, scale: float = 1.0) -> float:
    x = _c(x)
    return lib().oracle_lse(x.ctypes.data, _elem_dtype(x), 0, x.size, scale)


def jsd(x: np.ndarray, y: np.ndarray) -> float:
    x, y = _c(x), _c(y)
    assert x.dtype == y.dtype and x.size == y.size
    return lib().oracle_jsd(x.ctypes.data, y.ctypes.data, _elem_dtype(x), 0, 0, x.size)


def fused_argmax_near(a, b, t, beta: float, delta_source: int = 0):
    """The delta-fusion token of one row, argmax_k (t_k + beta * delta_k) taken exactly (lowest
    index on ties), and whether another entry lies within single-precision rounding of it."""
    a, b, t = _c(a), _c(b), _c(t)
    near = C.c_int(0)
    k = lib().oracle_fused_argmax_exact(a.ctypes.data, b.ctypes.data, t.ctypes.data, _elem_dtype(a), 0, a.size,
                                        float(np.float32(beta)), int(delta_source), C.byref(near))
    return k, bool(near.value)


def fused_argmax(a, b, t, beta: float) -> int:
    return fused_argmax_near(a, b, t, beta)[0]


def fused_argmax_fp32(a, b, t, beta: float, delta_source: int = 0) -> int:
    """What a single-precision evaluation of the same score picks (informational: the tests count
    the rows where it differs from the exact argmax, each of which must be a near tie)."""
    a, b, t = _c(a), _c(b), _c(t)
    return lib().oracle_fused_argmax_fp32(a.ctypes.data, b.ctypes.data, t.ctypes.data, _elem_dtype(a), 0, a.size,
                                          beta, int(delta_source))


# ------------------------------------------------------------------ AsymSpec

@dataclass
class AsymSpecResult:
    accept_len: np.ndarray   # [B] int32
    tokens: np.ndarray       # [B, K+1] int32
    D: np.ndarray            # [B, K+1] float64
    lse: np.ndarray          # [B, K+1, 3] float64 (a, b, t)
    margin: np.ndarray       # [B, K] float64
    argmax: np.ndarray       # [B, K+1] int32 (exact delta-fusion argmax of every row)
    flags: np.ndarray        # [B] uint32
    near: np.ndarray = None  # [B, K+1] bool: the row's argmax is a near tie


DELTA_A_MINUS_B = 0
DELTA_A = 1
DELTA_T_MINUS_B = 2


def fused_argmax_src(a, b, t, beta: float, delta_source: int) -> int:
    return fused_argmax_near(a, b, t, beta, delta_source)[0]


def asymspec_verify(a, b, t, draft_ids, beta: float, gamma: float, delta_source: int = 0) -> AsymSpecResult:
    a, b, t = _c(a), _c(b), _c(t)
    B, R, V = a.shape
    K = R - 1
    d = _c(np.asarray(draft_ids, np.int32).reshape(B, K))
    out = AsymSpecResult(np.zeros(B, np.int32), np.zeros((B, R), np.int32), np.zeros((B, R)),
                         np.zeros((B, R, 3)), np.zeros((B, max(K, 0))), np.zeros((B, R), np.int32),
                         np.zeros(B, np.uint32))
    near = np.zeros((B, R), np.int32)
    lib().oracle_asymspec_verify_src(a.ctypes.data, b.ctypes.data, t.ctypes.data, _elem_dtype(a), _p(d, C.c_int32),
                                     B, K, V, beta, gamma, delta_source, _p(out.accept_len, C.c_int32),
                                     _p(out.tokens, C.c_int32),
                                     _p(out.D, C.c_double), _p(out.lse, C.c_double), _p(out.margin, C.c_double),
                                     _p(out.argmax, C.c_int32), _p(near, C.c_int32), _p(out.flags, C.c_uint32))
    out.near = near.astype(bool)
    return out


# ------------------------------------------------------------------ Philox / RAPID

def philox4x32_10(ctr, key):
    c = np.asarray(ctr, np.uint32).copy()
    k = np.asarray(key, np.uint32).copy()
    o = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_p(c, C.c_uint32), _p(k, C.c_uint32), _p(o, C.c_uint32))
    return o


def uniform_from_word(w: int) -> float:
    return lib().oracle_uniform_from_word(int(w) & 0xFFFFFFFF)


def rapid_uniform(seed, offset, stream, req, row, word) -> float:
    return lib().oracle_rapid_uniform(seed, offset, stream, req, row, word)


@dataclass
class RapidRow:
    p: np.ndarray
    zhat: np.ndarray
    phat: np.ndarray
    prot: np.ndarray
    ntail: int
    near: bool


def rapid_row(z, q, T: float, eta: float, tail_frac: float = 0.1, tail_mode: int = 0) -> RapidRow:
    z = _c(np.asarray(z, np.float32))
    q = _c(np.asarray(q, np.float32))
    V = z.size
    p, zh, ph, pr = (np.zeros(V) for _ in range(4))
    near = C.c_int(0)
    n = lib().oracle_rapid_row_mode(_p(z, C.c_float), _p(q, C.c_float), V, T, eta, tail_frac, tail_mode,
                                    _p(p, C.c_double), _p(zh, C.c_double), _p(ph, C.c_double), _p(pr, C.c_double),
                                    C.byref(near))
    return RapidRow(p, zh, ph, pr, n, bool(near.value))


def race(w, seed, offset, stream, req, row):
    w = _c(np.asarray(w, np.float64))
    near = C.c_int(0)
    k = lib().oracle_race(_p(w, C.c_double), w.size, seed, offset, stream, req, row, C.byref(near))
    return k, bool(near.value)


@dataclass
class RapidResult:
    accept_len: np.ndarray
    tokens: np.ndarray
    flags: np.ndarray


def rapid_verify(z, q, draft_ids, T: float, eta: float, tail_frac: float, seed: int, offset: int = 0,
                 tail_mode: int = 0) -> RapidResult:
    z = _c(np.asarray(z, np.float32))
    q = _c(np.asarray(q, np.float32))
    B, R, V = z.shape
    G = R - 1
    d = _c(np.asarray(draft_ids, np.int32).reshape(B, G))
    out = RapidResult(np.zeros(B, np.int32), np.zeros((B, R), np.int32), np.zeros(B, np.uint32))
    lib().oracle_rapid_verify_mode(_p(z, C.c_float), _p(q, C.c_float), _p(d, C.c_int32), B, G, V, T, eta,
                                   tail_frac, tail_mode, seed, offset, _p(out.accept_len, C.c_int32),
                                   _p(out.tokens, C.c_int32), _p(out.flags, C.c_uint32))
    return out


# ------------------------------------------------------------------ E2-SCI

class SciStateC(C.Structure):
    """Per-request stabiliser state (T_applied, age, flags: 1 set, 2 fallback pending)."""
    _fields_ = [("T_applied", C.c_double), ("age", C.c_int32), ("flags", C.c_uint32)]


@dataclass(frozen=True)
class SciStabilisers:
    """E2-SCI stabilisers: hysteresis band, minimum refresh interval (windows), and the fallback to
    a conservative threshold after a window whose acceptance rate is below fallback_acc."""
    hysteresis: float = 0.0
    min_refresh: int = 1
    fallback_acc: float = 0.0
    fallback_T: float = 0.1


def sci_state(B: int):
    """A zero-filled stabiliser state array for B requests (before the first window)."""
    return (SciStateC * B)()


def sci_stab_threshold(state: "SciStateC", T_cand: float, s: SciStabilisers):
    """One window's threshold from the candidate and the state; returns (T_used, new_age)."""
    age = C.c_int32(0)
    T = lib().oracle_sci_stab_threshold(C.byref(state), T_cand, s.hysteresis, s.min_refresh, s.fallback_T,
                                        C.byref(age))
    return T, age.value


@dataclass(frozen=True)
class SciParams:
    T_base: float = 0.3
    alpha_omega: float = 0.2
    tau_credit: float = 0.6
    T_min: float = 0.1
    T_max: float = 0.6
    ewma_beta: float = 0.3


def sci_threshold(r_hat: float, p: SciParams = SciParams()) -> float:
    return lib().oracle_sci_threshold(r_hat, p.T_base, p.alpha_omega, p.tau_credit, p.T_min, p.T_max)


def sci_ewma(r_hat: float, p_acc: float, beta: float = 0.3) -> float:
    return lib().oracle_sci_ewma(r_hat, p_acc, beta)


@dataclass
class SciResult:
    accept_len: np.ndarray
    tokens: np.ndarray
    jsd: np.ndarray
    T: np.ndarray
    r_hat: np.ndarray
    flags: np.ndarray


def sci_verify(draft, target, draft_ids, r_hat, p: SciParams = SciParams(), stab: "SciStabilisers" = None,
               state=None) -> SciResult:
    """One window per request; with `stab`, `state` (from sci_state) is read and updated in place."""
    draft, target = _c(draft), _c(target)
    B, R, V = draft.shape
    K = R - 1
    d = _c(np.asarray(draft_ids, np.int32).reshape(B, K))
    rh = np.array(r_hat, np.float64, copy=True).reshape(B)
    out = SciResult(np.zeros(B, np.int32), np.zeros((B, R), np.int32), np.zeros((B, R)), np.zeros(B), rh,
                    np.zeros(B, np.uint32))
    if stab is None:
        lib().oracle_sci_verify(draft.ctypes.data, target.ctypes.data, _elem_dtype(draft), _p(d, C.c_int32), B, K,
                                V, p.T_base, p.alpha_omega, p.tau_credit, p.T_min, p.T_max, p.ewma_beta,
                                _p(rh, C.c_double), _p(out.accept_len, C.c_int32), _p(out.tokens, C.c_int32),
                                _p(out.jsd, C.c_double), _p(out.T, C.c_double), _p(out.flags, C.c_uint32))
        return out
    if state is None or len(state) != B:
        raise ValueError("stabilisers need a state array of B entries (sci_state(B))")
    lib().oracle_sci_verify_stab(draft.ctypes.data, target.ctypes.data, _elem_dtype(draft), _p(d, C.c_int32), B, K, V,
                                 p.T_base, p.alpha_omega, p.tau_credit, p.T_min, p.T_max, p.ewma_beta,
                                 stab.hysteresis, int(stab.min_refresh), stab.fallback_acc, stab.fallback_T, state,
                                 _p(rh, C.c_double), _p(out.accept_len, C.c_int32), _p(out.tokens, C.c_int32),
                                 _p(out.jsd, C.c_double), _p(out.T, C.c_double), _p(out.flags, C.c_uint32))
    return out
