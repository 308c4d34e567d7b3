"""Whole-batch grading of the full-size workloads against the oracle, on every host core.

Each worker process (started with `spawn`, before or independently of any GPU work in the
parent) generates its share of a batch's requests from the workload's seed -- the generator
keys every request by (seed, recipe, request index), so a share is the same bytes the whole
batch holds -- runs the oracle over them, and hands back both the inputs and the oracle's
results.  The parent assembles the batch for the GPU from the returned shares, so every request
is generated once.  Nothing here touches the GPU.
"""
from __future__ import annotations

import math
import multiprocessing as mp
import os
from dataclasses import dataclass, field

import numpy as np

import gen
import oracle


def host_pool(processes: int | None = None):
    """A spawn-started process pool over the host cores (the oracle library is built first, in the
    parent, so that workers only load it)."""
    oracle.lib()
    n = processes or os.cpu_count() or 1
    return mp.get_context("spawn").Pool(n)


def request_chunks(B: int, n_chunks: int):
    step = max(1, math.ceil(B / max(1, n_chunks)))
    return [list(range(s, min(B, s + step))) for s in range(0, B, step)]


# ------------------------------------------------------------------ workers


def _fp32_argmax_differs(batch, ref, beta, delta_source=0):
    """Rows where a single-precision evaluation of the delta-fusion score picks another entry than
    the exact argmax: (count, count of those the oracle marked near)."""
    n = d_near = 0
    for r in range(batch.a.shape[0]):
        for i in range(batch.a.shape[1]):
            k32 = oracle.fused_argmax_fp32(batch.a[r, i], batch.b[r, i], batch.t[r, i], beta, delta_source)
            if k32 != ref.argmax[r, i]:
                n += 1
                d_near += int(ref.near[r, i])
    return n, d_near


def asym_chunk(job):
    """Generate requests `reqs` of an AsymSpec batch and run the oracle for every (beta, gamma)."""
    recipe, seed, B, K, V, dtype, ident, reqs, runs, sci_r_hat = job
    batch = gen.make_asymspec_batch(recipe, seed, B, K, V, dtype, identical_frac=ident, requests=reqs)
    refs, differs = [], []
    seen_beta = {}
    for beta, gamma in runs:
        ref = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, beta, gamma)
        if beta not in seen_beta:   # the argmax depends on beta only
            seen_beta[beta] = _fp32_argmax_differs(batch, ref, beta)
        refs.append(ref)
        differs.append(seen_beta[beta])
    sci = None
    if sci_r_hat is not None:   # fused mode: the E2-SCI window on the same tensors (draft a, target t)
        sci = oracle.sci_verify(batch.a, batch.t, batch.drafts, np.asarray(sci_r_hat, np.float64))
    return reqs, (batch.a, batch.b, batch.t, batch.drafts, batch.identical), refs, differs, sci


def sci_chunk(job):
    """Generate requests `reqs` of one E2-SCI window and run the oracle from the given credit state."""
    recipe, seed, B, K, V, dtype, reqs, r_hat = job
    batch = gen.make_asymspec_batch(recipe, seed, B, K, V, dtype, requests=reqs)
    ref = oracle.sci_verify(batch.a, batch.t, batch.drafts, np.asarray(r_hat, np.float64))
    return reqs, (batch.a, batch.t, batch.drafts), ref


# ------------------------------------------------------------------ assembly


@dataclass
class AsymGraded:
    """A whole AsymSpec batch and the oracle's results for each run, over all requests."""
    a: np.ndarray
    b: np.ndarray
    t: np.ndarray
    drafts: np.ndarray
    identical: np.ndarray
    refs: list                      # per run: oracle.AsymSpecResult over all B requests
    fp32_differs: list              # per run: (rows where fp32 and exact argmax differ, of which near)
    sci: object = None              # fused mode: oracle.SciResult over all B requests


def _cat_results(parts, B, cls):
    """Concatenate per-chunk dataclass results (first axis = request) in request order."""
    out = {}
    for f in cls.__dataclass_fields__:
        vals = [getattr(p, f) for p in parts]
        if vals[0] is None:
            out[f] = None
        else:
            out[f] = np.concatenate(vals, axis=0)
    res = cls(**out)
    for f in cls.__dataclass_fields__:
        v = getattr(res, f)
        assert v is None or v.shape[0] == B, (f, v.shape, B)
    return res


def grade_asymspec_batch(pool, w, runs, seed=None, sci_r_hat=None, chunks_per_proc=4):
    """Generate workload `w` in the pool's workers and run the oracle over every request."""
    seed = w.seed if seed is None else seed
    ident = w.params.get("identical_frac", 0.0)
    n = (pool._processes or 1) * chunks_per_proc
    groups = request_chunks(w.B, n)
    jobs = [(w.recipe, seed, w.B, w.K, w.V, w.dtype, ident, g, runs,
             None if sci_r_hat is None else np.asarray(sci_r_hat)[g]) for g in groups]
    el = np.float32 if w.dtype == gen.F32 else np.uint16
    shape = (w.B, w.K + 1, w.V)
    a, b, t = (np.empty(shape, el) for _ in range(3))
    drafts = np.empty((w.B, w.K), np.int32)
    identical = np.zeros(w.B, bool)
    parts = {}
    for reqs, arrs, refs, differs, sci in pool.imap_unordered(asym_chunk, jobs):
        lo, hi = reqs[0], reqs[-1] + 1
        a[lo:hi], b[lo:hi], t[lo:hi], drafts[lo:hi], identical[lo:hi] = arrs
        parts[lo] = (refs, differs, sci)
    order = sorted(parts)
    refs = [_cat_results([parts[k][0][j] for k in order], w.B, oracle.AsymSpecResult) for j in range(len(runs))]
    differs = [tuple(sum(parts[k][1][j][m] for k in order) for m in range(2)) for j in range(len(runs))]
    sci = _cat_results([parts[k][2] for k in order], w.B, oracle.SciResult) if sci_r_hat is not None else None
    return AsymGraded(a, b, t, drafts, identical, refs, differs, sci)


def grade_sci_window(pool, w, seed, r_hat, chunks_per_proc=4):
    """One E2-SCI window of workload `w` (seed `seed`) from the oracle credit state `r_hat` [B]:
    returns (draft a, target t, drafts, oracle.SciResult over all B requests)."""
    n = (pool._processes or 1) * chunks_per_proc
    groups = request_chunks(w.B, n)
    jobs = [(w.recipe, seed, w.B, w.K, w.V, w.dtype, g, np.asarray(r_hat)[g]) for g in groups]
    el = np.float32 if w.dtype == gen.F32 else np.uint16
    shape = (w.B, w.K + 1, w.V)
    a, t = np.empty(shape, el), np.empty(shape, el)
    drafts = np.empty((w.B, w.K), np.int32)
    parts = {}
    for reqs, arrs, ref in pool.imap_unordered(sci_chunk, jobs):
        lo, hi = reqs[0], reqs[-1] + 1
        a[lo:hi], t[lo:hi], drafts[lo:hi] = arrs
        parts[lo] = ref
    ref = _cat_results([parts[k] for k in sorted(parts)], w.B, oracle.SciResult)
    return a, t, drafts, ref


# ------------------------------------------------------------------ comparison


@dataclass
class Tally:
    graded: int = 0
    flagged: int = 0
    notes: list = field(default_factory=list)


def compare_requests(acc, tok, st, ref_acc, ref_tok, ref_flags, tally: Tally, what: str):
    """Accept lengths and tokens bit-exact on every request the oracle does not flag; status bits
    (non-finite, bad draft) equal on all."""
    np.testing.assert_array_equal(st & 3, ref_flags & 3, err_msg=what)
    assert not (st & 4).any(), f"{what}: a bounded wait expired"
    ok = (ref_flags & oracle.FLAGS_UNGRADED) == 0
    tally.graded += int(ok.sum())
    tally.flagged += int((~ok).sum())
    bad = np.nonzero(ok & (acc != ref_acc))[0]
    assert bad.size == 0, f"{what}: accept length differs at requests {bad[:10]}"
    bad = np.nonzero(ok & np.any(tok != ref_tok, axis=1))[0]
    assert bad.size == 0, f"{what}: tokens differ at requests {bad[:10]}"
