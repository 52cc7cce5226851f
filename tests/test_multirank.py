"""Multi-rank host logic on CPU (gloo, world size 2).

Tokens are independent given (ids, req, local, ngram_context), so a batch
shards across ranks by token ranges with no exchange: a request cut at a
shard boundary continues with a carried context row (the last N-1 ids before
the cut).  Each rank hashes its shard with the oracle, the shards are
gathered, and the result must equal the unsharded batch.  The benchmark's
max-over-ranks timing reduction is exercised on the same process group.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rows(batch):
    import oracle
    req, local = oracle.token_index(batch.cu_seqlens, batch.num_requests, batch.num_tokens,
                                    batch.is_decode)
    return oracle.row_ids(batch.ids, req, local, batch.ngram_context, batch.layer_multipliers,
                          batch.vocab_sizes, batch.offsets, batch.ngram_size,
                          batch.heads_per_ngram, batch.boundary_id)


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import workloads as wl

    d = bench.Dist("gloo")
    try:
        for make in (wl.ragged_16, wl.mixed_8192, lambda: wl.decode(8)):
            full = make()
            T = full.num_tokens
            cut = [T * r // world for r in range(world + 1)]
            shard = wl.slice_batch(full, cut[rank], cut[rank + 1])
            mine = _rows(shard)
            gathered = [None] * world
            dist.all_gather_object(gathered, mine)
            if rank == 0:
                whole = np.concatenate(gathered, axis=1)
                results.put((full.name, bool(np.array_equal(whole, _rows(full)))))
        worst = d.max(float(rank + 1))
        if rank == 0:
            results.put(("max", worst == float(world)))
        d.barrier()
    finally:
        d.close()


def test_two_rank_shards_equal_the_whole_batch():
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = dict(results.get(timeout=10) for _ in range(4))
    assert got == {"ragged_16": True, "mixed_8192": True, "decode_b8": True, "max": True}, got


@pytest.mark.parametrize("cuts", [[0, 1, 29449], [0, 100, 5000, 29449], [0, 29448, 29449]])
def test_slices_at_any_cut_equal_the_whole_batch(cuts):
    sys.path.insert(0, ROOT)
    import workloads as wl
    full = wl.ragged_16()
    whole = _rows(full)
    parts = [_rows(wl.slice_batch(full, a, b)) for a, b in zip(cuts[:-1], cuts[1:])]
    assert np.array_equal(np.concatenate(parts, axis=1), whole)
