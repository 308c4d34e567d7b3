"""Host-side helpers for running the verification on several GPUs, one process per GPU.

Requests are independent (rows interact only inside a request's scan, and the E2-SCI
credit state is per request), so a batch shards over the request axis with no collective
on the data path: each rank verifies a contiguous block of requests on its own GPU.  The
only cross-rank steps are optional: gathering the small per-request outputs on the host,
and the max-over-ranks of a timing.
"""
from __future__ import annotations

from typing import List, Sequence


def request_shard(B: int, world_size: int, rank: int) -> slice:
    """Contiguous, balanced block of requests for `rank` (the first B % world_size ranks
    get one extra request)."""
    if world_size < 1 or not 0 <= rank < world_size or B < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(B, world_size)
    start = rank * base + min(rank, extra)
    return slice(start, start + base + (1 if rank < extra else 0))


def gather_rows(parts: Sequence, dim: int = 0):
    """Concatenate per-rank host tensors/arrays in rank order."""
    import numpy as np
    import torch
    if all(isinstance(p, torch.Tensor) for p in parts):
        return torch.cat(list(parts), dim=dim)
    return np.concatenate([np.asarray(p) for p in parts], axis=dim)


def all_gather_object_list(obj) -> List:
    """torch.distributed all_gather_object wrapper (identity when not distributed)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return [obj]
    out = [None] * dist.get_world_size()
    dist.all_gather_object(out, obj)
    return out


def max_over_ranks(x: float) -> float:
    """Largest value of `x` over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
