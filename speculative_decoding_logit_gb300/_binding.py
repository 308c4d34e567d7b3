"""ctypes binding to libasv.so: argument marshalling only (pointers, sizes, stream)."""
from __future__ import annotations

import ctypes as C
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

from . import nvcc_build as _build

ASV_F32 = 0
ASV_BF16 = 1
ASV_MODE_ASYMSPEC = 0
ASV_MODE_RAPID = 1
ASV_MODE_SCI = 2
REQ_NONFINITE = 1
REQ_BAD_DRAFT = 2
REQ_TIMEOUT = 4

_STATUS = {0: "ASV_OK", 1: "ASV_ERR_NULL", 2: "ASV_ERR_SHAPE", 3: "ASV_ERR_ALIGN", 4: "ASV_ERR_DTYPE",
           5: "ASV_ERR_PARAM", 6: "ASV_ERR_WORKSPACE", 7: "ASV_ERR_CUDA"}


class AsvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


_lib = None
_lib_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def library():
    """Load libasv.so (raises if it has not been built)."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise AsvError(-1, f"libasv.so not built ({_build.LIB}); call speculative_decoding_logit_gb300.build()")
            lib = C.CDLL(_build.LIB)
            _declare(lib)
            _lib = lib
    return _lib


_vp = C.c_void_p
_i = C.c_int
_sz = C.c_size_t
_f = C.c_float


class _AsymOptionsC(C.Structure):
    _fields_ = [("delta_source", C.c_int)]


DELTA_A_MINUS_B = 0
DELTA_A = 1
DELTA_T_MINUS_B = 2


class _RapidOptionsC(C.Structure):
    _fields_ = [("tail_mode", C.c_int)]


class _SciStabC(C.Structure):
    _fields_ = [("hysteresis", C.c_double), ("min_refresh", C.c_int32), ("reserved", C.c_int32),
                ("fallback_acc", C.c_double), ("fallback_T", C.c_double)]


class _SciParamsC(C.Structure):
    _fields_ = [("T_base", C.c_double), ("alpha_omega", C.c_double), ("tau_credit", C.c_double),
                ("T_min", C.c_double), ("T_max", C.c_double), ("ewma_beta", C.c_double)]


def _declare(L):
    L.asv_status_string.argtypes = [_i]
    L.asv_status_string.restype = C.c_char_p
    L.asv_last_cuda_error.argtypes = []
    L.asv_last_cuda_error.restype = _i
    L.asv_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
    L.asv_workspace_bytes.restype = _sz
    L.asv_workspace_init.argtypes = [_vp, _sz, _vp]
    L.asv_workspace_init.restype = _i
    L.asv_set_tuning.argtypes = [_i, _i]
    L.asv_set_tuning.restype = _i
    L.asv_set_kernel.argtypes = [_i]
    L.asv_set_kernel.restype = _i
    L.asv_query_plan.argtypes = [_i, _i, _i, _i, _i] + [C.POINTER(_i)] * 5
    L.asv_query_plan.restype = _i
    L.asymspec_verify.argtypes = [_vp, _vp, _vp, _i, _vp, _i, _i, _i, _f, _f, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
    L.asymspec_verify.restype = _i
    L.asymspec_verify_ex.argtypes = [_vp, _vp, _vp, _i, _vp, _i, _i, _i, _f, _f, C.POINTER(_AsymOptionsC), _vp, _vp,
                                     _vp, _vp, _vp, _vp, _sz, _vp]
    L.asymspec_verify_ex.restype = _i
    L.asv_host_arena_bytes.argtypes = [_i, _i, _i, _i]
    L.asv_host_arena_bytes.restype = _sz
    L.asymspec_verify_host.argtypes = [_vp, _vp, _vp, _i, _vp, _i, _i, _i, _f, _f, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
    L.asymspec_verify_host.restype = _i
    L.rapid_verify.argtypes = [_vp, _vp, _vp, _i, _i, _i, _f, _f, _f, C.c_uint64, C.c_uint32, _vp, _vp, _vp, _vp,
                               _sz, _vp]
    L.rapid_verify.restype = _i
    L.sci_verify.argtypes = [_vp, _vp, _i, _vp, _i, _i, _i, C.POINTER(_SciParamsC), _vp, _vp, _vp, _vp, _vp, _vp,
                             _vp, _sz, _vp]
    L.sci_verify.restype = _i
    L.asymspec_verify_sweep.argtypes = [_vp, _vp, _vp, _i, _vp, _i, _i, _i, C.POINTER(_f), _i, C.POINTER(_f), _i,
                                        _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
    L.asymspec_verify_sweep.restype = _i
    L.asymspec_sci_verify.argtypes = [_vp, _vp, _vp, _i, _vp, _i, _i, _i, _f, _f, C.POINTER(_SciParamsC), _vp, _vp,
                                      _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
    L.asymspec_sci_verify.restype = _i
    L.sci_verify_prehit.argtypes = [_vp, _vp, _i, _vp, _i, _i, _i, C.POINTER(_SciParamsC), _vp, _vp, _vp, _vp, _vp,
                                    _vp, _vp, _sz, _vp]
    L.sci_verify_prehit.restype = _i
    L.rapid_verify_ex.argtypes = [_vp, _vp, _vp, _i, _i, _i, _f, _f, _f, C.c_uint64, C.c_uint32,
                                  C.POINTER(_RapidOptionsC), _vp, _vp, _vp, _vp, _sz, _vp]
    L.rapid_verify_ex.restype = _i
    L.sci_verify_ex.argtypes = [_vp, _vp, _i, _vp, _i, _i, _i, C.POINTER(_SciParamsC), C.POINTER(_SciStabC), _vp,
                                _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
    L.sci_verify_ex.restype = _i


def _check(status: int, what: str):
    if status != 0:
        L = library()
        msg = L.asv_status_string(status).decode()
        if status == 7:
            msg += f" (cudaError {L.asv_last_cuda_error()})"
        raise AsvError(status, f"{what}: {msg}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream_handle(device: torch.device, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return ASV_F32
    if t.dtype == torch.bfloat16:
        return ASV_BF16
    raise AsvError(4, f"logits must be float32 or bfloat16, got {t.dtype}")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise AsvError(-1, "inputs must be CUDA tensors (the library has no CPU path)")


def _contig(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_contiguous():
        raise AsvError(2, f"{name} must be contiguous")
    return t


# Workspace cache: one zero-initialised buffer per (device, stream); every call leaves it zeroed.
_ws_cache: dict = {}
_ws_lock = threading.Lock()


def _workspace(device: torch.device, stream_handle: int, nbytes: int) -> torch.Tensor:
    key = (device.index, stream_handle)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.zeros(max(nbytes, 4096), dtype=torch.uint8, device=device)
            _ws_cache[key] = ws
    return ws


def workspace_bytes(mode: int, B: int, K: int, V: int, dtype: int) -> int:
    return int(library().asv_workspace_bytes(mode, B, K, V, dtype))


def set_tuning(cluster_ctas: int = 0, threads_per_cta: int = 0):
    _check(library().asv_set_tuning(cluster_ctas, threads_per_cta), "asv_set_tuning")


KERNEL_DEFAULT = 0
KERNEL_CLUSTER = 1
KERNEL_STAGED = 2


def set_kernel(which: int):
    """Kernel for later AsymSpec / E2-SCI calls: KERNEL_DEFAULT / KERNEL_CLUSTER (the cluster
    kernel) or KERNEL_STAGED (the staged kernel, where it applies)."""
    _check(library().asv_set_kernel(int(which)), "asv_set_kernel")


def query_plan(mode: int, B: int, K: int, V: int, dtype: int) -> dict:
    out = [C.c_int(0) for _ in range(5)]
    _check(library().asv_query_plan(mode, B, K, V, dtype, *[C.byref(o) for o in out]), "asv_query_plan")
    return {"cluster": out[0].value, "threads": out[1].value, "smem": out[2].value, "bulk": out[3].value,
            "max_active_clusters": out[4].value}


# ------------------------------------------------------------------ AsymSpec

@dataclass
class AsymSpecOutput:
    accept_len: torch.Tensor   # [B] int32
    tokens: torch.Tensor       # [B, K+1] int32, -1 padded
    D: torch.Tensor            # [B, K+1] float32
    lse: torch.Tensor          # [B, K+1, 3] float32 (a, b, t)
    req_status: torch.Tensor   # [B] int32 (ASV_REQ_* bits)


def asymspec_verify(a: torch.Tensor, b: torch.Tensor, t: torch.Tensor, draft_ids: torch.Tensor,
                    beta: float = 1.0, gamma: float = 0.5, *, delta_source: int = DELTA_A_MINUS_B,
                    out: Optional[AsymSpecOutput] = None, workspace: Optional[torch.Tensor] = None,
                    stream=None) -> AsymSpecOutput:
    """AsymSpec verification of a [B, K+1, V] batch (see include/asv.h).  `delta_source`
    selects the context-gain signal of the delta-fusion score (asymspec_verify_ex)."""
    _need_cuda(a, b, t, draft_ids)
    if a.dim() != 3 or a.shape != b.shape or a.shape != t.shape:
        raise AsvError(2, "a, b, t must share one [B, K+1, V] shape")
    if a.dtype != b.dtype or a.dtype != t.dtype:
        raise AsvError(4, "a, b, t must share one dtype")
    B, R1, V = a.shape
    K = R1 - 1
    if draft_ids.dtype != torch.int32 or tuple(draft_ids.shape) != (B, K):
        raise AsvError(2, "draft_ids must be int32 [B, K]")
    for n, x in (("a", a), ("b", b), ("t", t), ("draft_ids", draft_ids)):
        _contig(x, n)
    dev = a.device
    sh = _stream_handle(dev, stream)
    if out is None:
        out = AsymSpecOutput(torch.empty(B, dtype=torch.int32, device=dev),
                             torch.empty(B, R1, dtype=torch.int32, device=dev),
                             torch.empty(B, R1, dtype=torch.float32, device=dev),
                             torch.empty(B, R1, 3, dtype=torch.float32, device=dev),
                             torch.empty(B, dtype=torch.int32, device=dev))
    dt = _dtype_code(a)
    need = workspace_bytes(ASV_MODE_ASYMSPEC, B, K, V, dt)
    ws = workspace if workspace is not None else _workspace(dev, sh, need)
    if delta_source == DELTA_A_MINUS_B:
        st = library().asymspec_verify(_ptr(a), _ptr(b), _ptr(t), dt, _ptr(draft_ids), B, K, V, float(beta),
                                       float(gamma), _ptr(out.accept_len), _ptr(out.tokens), _ptr(out.D),
                                       _ptr(out.lse), _ptr(out.req_status), _ptr(ws), ws.numel() * ws.element_size(),
                                       sh)
        _check(st, "asymspec_verify")
    else:
        opt = _AsymOptionsC(int(delta_source))
        st = library().asymspec_verify_ex(_ptr(a), _ptr(b), _ptr(t), dt, _ptr(draft_ids), B, K, V, float(beta),
                                          float(gamma), C.byref(opt), _ptr(out.accept_len), _ptr(out.tokens),
                                          _ptr(out.D), _ptr(out.lse), _ptr(out.req_status), _ptr(ws),
                                          ws.numel() * ws.element_size(), sh)
        _check(st, "asymspec_verify_ex")
    return out


def host_arena_bytes(B: int, K: int, V: int, dtype: int) -> int:
    return int(library().asv_host_arena_bytes(B, K, V, dtype))


ASV_MODE_SWEEP = 3
ASV_MODE_ASYMSPEC_SCI = 4


@dataclass
class SweepOutput:
    accept_len: torch.Tensor  # [n_gamma, B] int32
    tokens: torch.Tensor      # [n_beta, n_gamma, B, K+1] int32
    D: torch.Tensor           # [B, K+1] float32
    lse: torch.Tensor         # [B, K+1, 3] float32
    req_status: torch.Tensor  # [B] int32


def _check_asym_inputs(a, b, t, draft_ids):
    _need_cuda(a, b, t, draft_ids)
    if a.dim() != 3 or a.shape != b.shape or a.shape != t.shape:
        raise AsvError(2, "a, b, t must share one [B, K+1, V] shape")
    if a.dtype != b.dtype or a.dtype != t.dtype:
        raise AsvError(4, "a, b, t must share one dtype")
    B, R1, V = a.shape
    if draft_ids.dtype != torch.int32 or tuple(draft_ids.shape) != (B, R1 - 1):
        raise AsvError(2, "draft_ids must be int32 [B, K]")
    for n, x in (("a", a), ("b", b), ("t", t), ("draft_ids", draft_ids)):
        _contig(x, n)
    return B, R1 - 1, V


def asymspec_verify_sweep(a: torch.Tensor, b: torch.Tensor, t: torch.Tensor, draft_ids: torch.Tensor, betas,
                          gammas, *, workspace: Optional[torch.Tensor] = None, stream=None) -> SweepOutput:
    """AsymSpec for every (beta, gamma) of a grid from one read of a, b, t (asymspec_verify_sweep)."""
    B, K, V = _check_asym_inputs(a, b, t, draft_ids)
    betas = [float(x) for x in betas]
    gammas = [float(x) for x in gammas]
    nb, ng = len(betas), len(gammas)
    dev = a.device
    sh = _stream_handle(dev, stream)
    out = SweepOutput(torch.empty(ng, B, dtype=torch.int32, device=dev),
                      torch.empty(nb, ng, B, K + 1, dtype=torch.int32, device=dev),
                      torch.empty(B, K + 1, dtype=torch.float32, device=dev),
                      torch.empty(B, K + 1, 3, dtype=torch.float32, device=dev),
                      torch.empty(B, dtype=torch.int32, device=dev))
    dt = _dtype_code(a)
    ws = workspace if workspace is not None else _workspace(dev, sh, workspace_bytes(ASV_MODE_SWEEP, B, K, V, dt))
    bb = (_f * max(nb, 1))(*betas)
    gg = (_f * max(ng, 1))(*gammas)
    st = library().asymspec_verify_sweep(_ptr(a), _ptr(b), _ptr(t), dt, _ptr(draft_ids), B, K, V, bb, nb, gg, ng,
                                         _ptr(out.accept_len), _ptr(out.tokens), _ptr(out.D), _ptr(out.lse),
                                         _ptr(out.req_status), _ptr(ws), ws.numel(), sh)
    _check(st, "asymspec_verify_sweep")
    return out


@dataclass
class AsymSciOutput:
    accept_len: torch.Tensor      # AsymSpec [B]
    tokens: torch.Tensor          # AsymSpec [B, K+1]
    D: torch.Tensor               # JSD(a || b) [B, K+1]
    lse: torch.Tensor             # [B, K+1, 3]
    sci_accept_len: torch.Tensor  # E2-SCI [B]
    sci_tokens: torch.Tensor      # E2-SCI [B, K+1]
    jsd: torch.Tensor             # JSD(a || t) [B, K+1]
    T: torch.Tensor               # E2-SCI threshold [B]
    req_status: torch.Tensor      # [B]


def asymspec_sci_verify(a: torch.Tensor, b: torch.Tensor, t: torch.Tensor, draft_ids: torch.Tensor, beta: float,
                        gamma: float, r_hat: torch.Tensor, params: "SciParams" = None, *,
                        workspace: Optional[torch.Tensor] = None, stream=None) -> AsymSciOutput:
    """AsymSpec and one E2-SCI window (draft = a, target = t) from one read (asymspec_sci_verify);
    r_hat (float64 [B], device) is updated in place."""
    B, K, V = _check_asym_inputs(a, b, t, draft_ids)
    if r_hat.dtype != torch.float64 or tuple(r_hat.shape) != (B,) or not r_hat.is_cuda:
        raise AsvError(2, "r_hat must be a float64 [B] CUDA tensor")
    params = params or SciParams()
    dev = a.device
    sh = _stream_handle(dev, stream)
    i32 = lambda *sh_: torch.empty(*sh_, dtype=torch.int32, device=dev)
    f32 = lambda *sh_: torch.empty(*sh_, dtype=torch.float32, device=dev)
    out = AsymSciOutput(i32(B), i32(B, K + 1), f32(B, K + 1), f32(B, K + 1, 3), i32(B), i32(B, K + 1),
                        f32(B, K + 1), f32(B), i32(B))
    dt = _dtype_code(a)
    ws = workspace if workspace is not None else _workspace(dev, sh,
                                                            workspace_bytes(ASV_MODE_ASYMSPEC_SCI, B, K, V, dt))
    pc = _SciParamsC(params.T_base, params.alpha_omega, params.tau_credit, params.T_min, params.T_max,
                     params.ewma_beta)
    st = library().asymspec_sci_verify(_ptr(a), _ptr(b), _ptr(t), dt, _ptr(draft_ids), B, K, V, float(beta),
                                       float(gamma), C.byref(pc), _ptr(r_hat), _ptr(out.accept_len), _ptr(out.tokens),
                                       _ptr(out.D), _ptr(out.lse), _ptr(out.sci_accept_len), _ptr(out.sci_tokens),
                                       _ptr(out.jsd), _ptr(out.T), _ptr(out.req_status), _ptr(ws), ws.numel(), sh)
    _check(st, "asymspec_sci_verify")
    return out


def asymspec_verify_host(a, b, t, draft_ids, beta, gamma, arena: torch.Tensor, out_accept_len, out_tokens, out_D,
                         out_req_status, dtype: int, stream=None):
    """AsymSpec verification over host (pinned) buffers: raw addresses of CPU tensors; `arena`
    is a zeroed device uint8 tensor of host_arena_bytes() bytes.  Asynchronous on the stream."""
    B, R1, V = a.shape
    K = R1 - 1
    sh = _stream_handle(arena.device, stream)
    st = library().asymspec_verify_host(_ptr(a), _ptr(b), _ptr(t), dtype, _ptr(draft_ids), B, K, V, float(beta),
                                        float(gamma), _ptr(out_accept_len), _ptr(out_tokens), _ptr(out_D),
                                        _ptr(out_req_status), _ptr(arena), arena.numel(), sh)
    _check(st, "asymspec_verify_host")


# ------------------------------------------------------------------ RAPID

@dataclass
class RapidOutput:
    accept_len: torch.Tensor
    tokens: torch.Tensor
    req_status: torch.Tensor


TAIL_KEEP_P = 0          # tail entries keep p, the head is rescaled (rapid_verify's reading)
TAIL_RENORMALISE_ALL = 1  # p substitutes phat on the tail, then every entry is renormalised


def rapid_verify(z: torch.Tensor, q: torch.Tensor, draft_ids: torch.Tensor, T: float = 1.0, eta: float = 10.0,
                 tail_frac: float = 0.1, seed: int = 1234, offset: int = 0, *, tail_mode: int = TAIL_KEEP_P,
                 out: Optional[RapidOutput] = None, workspace: Optional[torch.Tensor] = None,
                 stream=None) -> RapidOutput:
    """RAPID verification of fp32 target logits z and drafter probabilities q, [B, G+1, V]
    (`tail_mode` selects the reading of the tail protection, see rapid_verify_ex)."""
    _need_cuda(z, q, draft_ids)
    if z.dim() != 3 or z.shape != q.shape:
        raise AsvError(2, "z and q must share one [B, G+1, V] shape")
    if z.dtype != torch.float32 or q.dtype != torch.float32:
        raise AsvError(4, "RAPID takes float32 z and q")
    B, R1, V = z.shape
    G = R1 - 1
    if draft_ids.dtype != torch.int32 or tuple(draft_ids.shape) != (B, G):
        raise AsvError(2, "draft_ids must be int32 [B, G]")
    for n, x in (("z", z), ("q", q), ("draft_ids", draft_ids)):
        _contig(x, n)
    dev = z.device
    sh = _stream_handle(dev, stream)
    if out is None:
        out = RapidOutput(torch.empty(B, dtype=torch.int32, device=dev),
                          torch.empty(B, R1, dtype=torch.int32, device=dev),
                          torch.empty(B, dtype=torch.int32, device=dev))
    need = workspace_bytes(ASV_MODE_RAPID, B, G, V, ASV_F32)
    ws = workspace if workspace is not None else _workspace(dev, sh, need)
    opt = _RapidOptionsC(int(tail_mode))
    st = library().rapid_verify_ex(_ptr(z), _ptr(q), _ptr(draft_ids), B, G, V, float(T), float(eta),
                                   float(tail_frac), int(seed) & 0xFFFFFFFFFFFFFFFF, int(offset) & 0xFFFFFFFF,
                                   C.byref(opt), _ptr(out.accept_len), _ptr(out.tokens), _ptr(out.req_status),
                                   _ptr(ws), ws.numel(), sh)
    _check(st, "rapid_verify_ex")
    return out


# ------------------------------------------------------------------ E2-SCI

@dataclass(frozen=True)
class SciParams:
    T_base: float = 0.3
    alpha_omega: float = 0.2
    tau_credit: float = 0.6
    T_min: float = 0.1
    T_max: float = 0.6
    ewma_beta: float = 0.3


@dataclass
class SciOutput:
    accept_len: torch.Tensor
    tokens: torch.Tensor
    jsd: torch.Tensor
    T: torch.Tensor
    req_status: torch.Tensor


@dataclass(frozen=True)
class SciStabilisers:
    """E2-SCI stabilisers (see sci_verify_ex in include/asv.h)."""
    hysteresis: float = 0.0
    min_refresh: int = 1
    fallback_acc: float = 0.0
    fallback_T: float = 0.1


def sci_state_new(B: int, device="cuda") -> torch.Tensor:
    """Zero-filled stabiliser state for B requests: [B, 4] int32 (16 bytes per request: T_applied
    as float64, then age and flags)."""
    return torch.zeros(B, 4, dtype=torch.int32, device=device)


def sci_state_decode(state: torch.Tensor):
    """(T_applied float64 [B], age int32 [B], flags int32 [B]) of a state tensor (copied to host)."""
    h = state.cpu().contiguous()
    return h[:, :2].contiguous().view(torch.float64).reshape(-1), h[:, 2].clone(), h[:, 3].clone()


def sci_verify(draft: torch.Tensor, target: torch.Tensor, draft_ids: torch.Tensor, r_hat: torch.Tensor,
               params: SciParams = SciParams(), *, stabilisers: Optional[SciStabilisers] = None,
               state: Optional[torch.Tensor] = None, prehit: bool = False, out: Optional[SciOutput] = None,
               workspace: Optional[torch.Tensor] = None, stream=None) -> SciOutput:
    """One E2-SCI window; r_hat (float64 [B], device) is updated in place, and with `stabilisers`
    so is `state` (from sci_state_new).  `prehit` verifies every window's first draft first and
    drops windows whose first draft fails (sci_verify_prehit; no stabilisers)."""
    _need_cuda(draft, target, draft_ids, r_hat)
    if draft.dim() != 3 or draft.shape != target.shape or draft.dtype != target.dtype:
        raise AsvError(2, "draft and target must share one [B, K+1, V] shape and dtype")
    B, R1, V = draft.shape
    K = R1 - 1
    if draft_ids.dtype != torch.int32 or tuple(draft_ids.shape) != (B, K):
        raise AsvError(2, "draft_ids must be int32 [B, K]")
    if r_hat.dtype != torch.float64 or tuple(r_hat.shape) != (B,):
        raise AsvError(2, "r_hat must be float64 [B]")
    for n, x in (("draft", draft), ("target", target), ("draft_ids", draft_ids), ("r_hat", r_hat)):
        _contig(x, n)
    if stabilisers is not None:
        if state is None or state.dtype != torch.int32 or tuple(state.shape) != (B, 4) or not state.is_cuda:
            raise AsvError(2, "state must be an int32 [B, 4] CUDA tensor (sci_state_new)")
        _contig(state, "state")
    dev = draft.device
    sh = _stream_handle(dev, stream)
    if out is None:
        out = SciOutput(torch.empty(B, dtype=torch.int32, device=dev),
                        torch.empty(B, R1, dtype=torch.int32, device=dev),
                        torch.empty(B, R1, dtype=torch.float32, device=dev),
                        torch.empty(B, dtype=torch.float32, device=dev),
                        torch.empty(B, dtype=torch.int32, device=dev))
    dt = _dtype_code(draft)
    need = workspace_bytes(ASV_MODE_SCI, B, K, V, dt)
    ws = workspace if workspace is not None else _workspace(dev, sh, need)
    pc = _SciParamsC(params.T_base, params.alpha_omega, params.tau_credit, params.T_min, params.T_max,
                     params.ewma_beta)
    if prehit:
        if stabilisers is not None:
            raise AsvError(5, "the pre-hit path takes no stabilisers")
        st = library().sci_verify_prehit(_ptr(draft), _ptr(target), dt, _ptr(draft_ids), B, K, V, C.byref(pc),
                                         _ptr(r_hat), _ptr(out.accept_len), _ptr(out.tokens), _ptr(out.jsd),
                                         _ptr(out.T), _ptr(out.req_status), _ptr(ws), ws.numel(), sh)
        _check(st, "sci_verify_prehit")
        return out
    if stabilisers is None:
        st = library().sci_verify(_ptr(draft), _ptr(target), dt, _ptr(draft_ids), B, K, V, C.byref(pc), _ptr(r_hat),
                                  _ptr(out.accept_len), _ptr(out.tokens), _ptr(out.jsd), _ptr(out.T),
                                  _ptr(out.req_status), _ptr(ws), ws.numel(), sh)
        _check(st, "sci_verify")
        return out
    sc = _SciStabC(float(stabilisers.hysteresis), int(stabilisers.min_refresh), 0, float(stabilisers.fallback_acc),
                   float(stabilisers.fallback_T))
    st = library().sci_verify_ex(_ptr(draft), _ptr(target), dt, _ptr(draft_ids), B, K, V, C.byref(pc), C.byref(sc),
                                 _ptr(r_hat), _ptr(state), _ptr(out.accept_len), _ptr(out.tokens), _ptr(out.jsd),
                                 _ptr(out.T), _ptr(out.req_status), _ptr(ws), ws.numel(), sh)
    _check(st, "sci_verify_ex")
    return out
