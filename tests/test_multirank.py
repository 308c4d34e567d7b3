"""World-size-2 gloo ranks on CPU: the request sharding, the host-side gather of per-request
outputs and the max-over-ranks timing reduction used by the multi-GPU benchmark.  Each rank's
verification is stood in for by the oracle (no GPU here); the concatenated shard results must
equal the full-batch result."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from speculative_decoding_logit_gb300.shard import request_shard


def test_request_shard_partitions():
    for B in (0, 1, 5, 64, 1023):
        for W in (1, 2, 3, 8):
            sl = [request_shard(B, W, r) for r in range(W)]
            covered = [i for s in sl for i in range(B)[s]]
            assert covered == list(range(B))
            sizes = [s.stop - s.start for s in sl]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        request_shard(4, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist

    import gen
    import oracle
    from speculative_decoding_logit_gb300.shard import all_gather_object_list, gather_rows, max_over_ranks
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        batch = gen.make_asymspec_batch("spiky", 5, 7, 2, 300, gen.BF16, identical_frac=0.3)
        sl = request_shard(batch.B, world, rank)
        res = oracle.asymspec_verify(batch.a[sl], batch.b[sl], batch.t[sl], batch.drafts[sl], 1.0, 0.5)
        parts = all_gather_object_list((res.accept_len, res.tokens, res.D))
        t = max_over_ranks(0.25 + rank)
        if rank == 0:
            full = oracle.asymspec_verify(batch.a, batch.b, batch.t, batch.drafts, 1.0, 0.5)
            acc = gather_rows([p[0] for p in parts])
            tok = gather_rows([p[1] for p in parts])
            D = gather_rows([p[2] for p in parts])
            ok = (np.array_equal(acc, full.accept_len) and np.array_equal(tok, full.tokens)
                  and np.array_equal(D, full.D) and t == 1.25)
            q.put(ok)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_gather():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    assert q.get() is True
