"""Seeded synthetic logit workloads for the verification step.

This module is shared by the CPU oracle tests, the CUDA parity tests and the
benchmark.  It holds random draws and storage rounding only: no log-softmax,
no divergence, no argmax over the verifier, no gate.  (The drafter's own greedy
choice, argmax of its logits, and the RAPID drafter's probability vector are
part of what a drafter hands to the verifier, so they are generated here.)

Every request is generated from its own PCG64 stream keyed by
``(seed, recipe, request index)``, so any single request can be regenerated
alone (the full-size parity tests rebuild sampled requests on the host) and a
large batch can be generated in parallel.

Storage: fp32 arrays are ``float32``; bf16 arrays are ``uint16`` bit patterns
(round-to-nearest-even from fp32), which ``torch`` can view as ``bfloat16``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

F32 = 0
BF16 = 1
DTYPE_NAMES = {F32: "f32", BF16: "bf16"}

# Recipe tags mixed into every seed sequence.
_TAG_SPIKY = 11
_TAG_GUMBEL_ZIPF = 12
_TAG_RAPID = 13
_TAG_IDENTICAL = 14

BASE_SEED = 20260827


# --------------------------------------------------------------------------- storage

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 exactly."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def store(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round float64 draws once to fp32, then (for bf16) to bf16."""
    x32 = np.asarray(x, dtype=np.float32)
    if dtype == F32:
        return x32
    if dtype == BF16:
        return f32_to_bf16_bits(x32)
    raise ValueError(f"unknown dtype {dtype}")


def widen(x: np.ndarray, dtype: int) -> np.ndarray:
    """Stored values as float32 (exact)."""
    return x if dtype == F32 else bf16_bits_to_f32(x)


def _rng(seed: int, *tags: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed) & 0xFFFFFFFF, *map(int, tags)])))


def _first_argmax(rows: np.ndarray) -> np.ndarray:
    # numpy's argmax returns the lowest index among equal maxima.
    return np.argmax(rows, axis=-1).astype(np.int32)


# --------------------------------------------------------------------------- recipes (one request)

def spiky_gaussian_request(seed: int, req: int, K: int, V: int, dtype: int, identical: bool = False):
    """One request of the Gaussian-with-spikes recipe.

    a ~ N(0, 2^2) per entry with +8 added at 5 distinct random ids per row,
    b = a + N(0, 0.5^2) (or b = a bitwise when ``identical``), t = b + N(0, 1^2);
    draft i = lowest argmax of the stored a_i, for i < K.
    """
    g = _rng(seed, _TAG_SPIKY, req)
    R = K + 1
    a = g.standard_normal((R, V)) * 2.0
    nspike = min(5, V)
    for r in range(R):
        ids = g.choice(V, size=nspike, replace=False)
        a[r, ids] += 8.0
    a_s = store(a, dtype)
    a_w = widen(a_s, dtype).astype(np.float64)
    if identical:
        b_s = a_s.copy()
        g.standard_normal((R, V))  # keep the stream position independent of the flag
    else:
        b_s = store(a_w + 0.5 * g.standard_normal((R, V)), dtype)
    b_w = widen(b_s, dtype).astype(np.float64)
    t_s = store(b_w + g.standard_normal((R, V)), dtype)
    drafts = _first_argmax(widen(a_s[:K], dtype)) if K > 0 else np.zeros((0,), np.int32)
    return a_s, b_s, t_s, drafts


def gumbel_zipf_request(seed: int, req: int, K: int, V: int, dtype: int = BF16):
    """One request of the Gumbel/Zipf recipe.

    a_k = 1.5 * Gumbel(0, 1) - 1.1 * ln(rank_k), rank_k the 1-based position of id k
    in a per-row random permutation (a Zipf(s=1.1) log-boost); b = a + N(0, 0.7^2)
    on a Bernoulli(0.2) mask of ids per row, b = a elsewhere; t = b + N(0, 1^2);
    draft i = lowest argmax of the stored a_i.
    """
    g = _rng(seed, _TAG_GUMBEL_ZIPF, req)
    R = K + 1
    a = np.empty((R, V))
    for r in range(R):
        rank = np.empty(V)
        rank[g.permutation(V)] = np.arange(1, V + 1)
        a[r] = 1.5 * g.gumbel(size=V) - 1.1 * np.log(rank)
    a_s = store(a, dtype)
    a_w = widen(a_s, dtype).astype(np.float64)
    mask = g.random((R, V)) < 0.2
    b = np.where(mask, a_w + 0.7 * g.standard_normal((R, V)), a_w)
    b_s = store(b, dtype)
    # Where the mask is off b is a bitwise copy of a.
    b_s = np.where(mask, b_s, a_s)
    b_w = widen(b_s, dtype).astype(np.float64)
    t_s = store(b_w + g.standard_normal((R, V)), dtype)
    drafts = _first_argmax(widen(a_s[:K], dtype)) if K > 0 else np.zeros((0,), np.int32)
    return a_s, b_s, t_s, drafts


def rapid_request(seed: int, req: int, G: int, V: int):
    """One request of the long-context retrieval-drafter recipe (fp32).

    Target logits z = N(0, 2^2) - 1.1 ln(rank); the drafter's probabilities are
    q = normalised exp(z + N(0, 1^2)) formed in float64 and stored in fp32 (not
    renormalised after rounding); draft i is sampled from q_i.
    """
    g = _rng(seed, _TAG_RAPID, req)
    R = G + 1
    z = np.empty((R, V))
    for r in range(R):
        rank = np.empty(V)
        rank[g.permutation(V)] = np.arange(1, V + 1)
        z[r] = 2.0 * g.standard_normal(V) - 1.1 * np.log(rank)
    z_s = store(z, F32)
    zq = z_s.astype(np.float64) + g.standard_normal((R, V))
    w = np.exp(zq - zq.max(axis=1, keepdims=True))
    qd = w / w.sum(axis=1, keepdims=True)
    q_s = qd.astype(np.float32)
    drafts = np.empty(G, np.int32)
    for i in range(G):
        c = np.cumsum(qd[i])
        drafts[i] = min(int(np.searchsorted(c, g.random() * c[-1], side="right")), V - 1)
    return z_s, q_s, drafts


# --------------------------------------------------------------------------- batches

@dataclass
class Batch:
    """A batch of requests laid out as [B, K+1, V] (rows contiguous) plus drafts [B, K]."""
    a: np.ndarray
    b: np.ndarray
    t: np.ndarray
    drafts: np.ndarray
    dtype: int
    B: int
    K: int
    V: int
    identical: Optional[np.ndarray] = None  # per request: b == a bitwise


@dataclass
class RapidBatch:
    z: np.ndarray
    q: np.ndarray
    drafts: np.ndarray
    B: int
    G: int
    V: int


def _alloc(shape, dtype, out=None):
    if out is not None:
        return out
    return np.empty(shape, np.float32 if dtype == F32 else np.uint16)


def identical_requests(seed: int, B: int, frac: float) -> np.ndarray:
    """Exactly round(frac*B) requests, chosen at random, get b = a bitwise."""
    g = _rng(seed, _TAG_IDENTICAL, B)
    mask = np.zeros(B, bool)
    mask[g.permutation(B)[: int(round(frac * B))]] = True
    return mask


def _spiky_worker(args):
    seed, reqs, K, V, dtype, ident = args
    return [spiky_gaussian_request(seed, r, K, V, dtype, bool(ident[i])) for i, r in enumerate(reqs)]


def _gz_worker(args):
    seed, reqs, K, V, dtype = args
    return [gumbel_zipf_request(seed, r, K, V, dtype) for r in reqs]


def _map_requests(worker, jobs, processes):
    if processes and processes > 1 and len(jobs) > 1:
        import multiprocessing as mp
        with mp.get_context("spawn").Pool(processes) as pool:
            return pool.map(worker, jobs)
    return [worker(j) for j in jobs]


def _chunks(B, n):
    step = max(1, math.ceil(B / max(1, n)))
    return [list(range(s, min(B, s + step))) for s in range(0, B, step)]


def make_asymspec_batch(recipe: str, seed: int, B: int, K: int, V: int, dtype: int,
                        identical_frac: float = 0.0, processes: int = 0, requests=None) -> Batch:
    """Build a batch; ``requests`` selects a subset of request indices (default all B)."""
    reqs = list(range(B)) if requests is None else [int(r) for r in requests]
    n = len(reqs)
    ident_all = identical_requests(seed, B, identical_frac) if identical_frac > 0 else np.zeros(B, bool)
    a = _alloc((n, K + 1, V), dtype)
    b = _alloc((n, K + 1, V), dtype)
    t = _alloc((n, K + 1, V), dtype)
    drafts = np.empty((n, K), np.int32)
    nproc = processes if n >= 8 else 0
    groups = _chunks(n, (nproc or 1) * 4)
    if recipe == "spiky":
        jobs = [(seed, [reqs[i] for i in grp], K, V, dtype, [ident_all[reqs[i]] for i in grp]) for grp in groups]
        res = _map_requests(_spiky_worker, jobs, nproc)
    elif recipe == "gumbel_zipf":
        jobs = [(seed, [reqs[i] for i in grp], K, V, dtype) for grp in groups]
        res = _map_requests(_gz_worker, jobs, nproc)
    else:
        raise ValueError(recipe)
    i = 0
    for part in res:
        for (ra, rb, rt, rd) in part:
            a[i], b[i], t[i], drafts[i] = ra, rb, rt, rd
            i += 1
    return Batch(a, b, t, drafts, dtype, n, K, V, ident_all[reqs])


def make_rapid_batch(seed: int, B: int, G: int, V: int, requests=None) -> RapidBatch:
    reqs = list(range(B)) if requests is None else [int(r) for r in requests]
    n = len(reqs)
    z = np.empty((n, G + 1, V), np.float32)
    q = np.empty((n, G + 1, V), np.float32)
    d = np.empty((n, G), np.int32)
    for i, r in enumerate(reqs):
        z[i], q[i], d[i] = rapid_request(seed, r, G, V)
    return RapidBatch(z, q, d, n, G, V)


# --------------------------------------------------------------------------- named workloads

@dataclass(frozen=True)
class Workload:
    name: str
    mode: str          # "asymspec", "rapid", "sci"
    recipe: str
    B: int
    K: int             # drafts per request (RAPID: gamma_draft)
    V: int
    dtype: int
    seed: int
    params: dict = field(default_factory=dict)


WORKLOADS = {
    w.name: w for w in [
        Workload("asymspec_b1_k2_v32000_f32", "asymspec", "spiky", 1, 2, 32000, F32, BASE_SEED + 1,
                 {"runs": [(1.0, 0.5)]}),
        Workload("asymspec_b64_k2_v151936_bf16", "asymspec", "gumbel_zipf", 64, 2, 151936, BF16, BASE_SEED + 2,
                 {"runs": [(1.0, 0.5), (0.0, 1.0)]}),
        Workload("asymspec_sweep_b256_k4_v151936_f32", "asymspec", "spiky", 256, 4, 151936, F32, BASE_SEED + 3,
                 {"runs": [(bb, gg) for bb in (0.0, 1.0, 1.5, 2.0) for gg in (0.4, 0.5, 0.7, 1.0)],
                  "identical_frac": 0.3}),
        Workload("rapid_b32_g10_v128256_f32", "rapid", "rapid", 32, 10, 128256, F32, 1234,
                 {"T": 1.0, "etas": [0.0, 5.0, 10.0, 20.0], "tail_frac": 0.1, "philox_seed": 1234}),
        Workload("sci_asymspec_b1024_k8_v151936_bf16", "sci", "spiky", 1024, 8, 151936, BF16, BASE_SEED + 5,
                 {"windows": 5, "r_hat0": 0.6, "ewma_beta": 0.3, "T_base": 0.3, "alpha_omega": 0.2,
                  "tau_credit": 0.6, "T_min": 0.1, "T_max": 0.6, "runs": [(1.0, 0.5)]}),
    ]
}
