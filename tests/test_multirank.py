"""Multi-rank host logic on CPU (gloo, world size 2 and 3).

Tokens are independent given (ids, req, local, ngram_context), so a batch
shards across ranks by token ranges with no exchange: a request cut at a
shard boundary continues with a carried context row (the last N-1 ids before
the cut).  Each rank takes its share from the library's planner
(ple_shard_plan, host code, runs without a GPU), builds its shard's
cu_seqlens and context rows from the oracle's definition of the carried
context, hashes the shard with the oracle, and the gathered rows must equal
the unsharded batch.  The benchmark's max-over-ranks timing reduction is
exercised on the same process group.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rows(ids, cu, ctx, batch, is_decode):
    import oracle
    T, B = ids.shape[0], ctx.shape[0]
    req, local = oracle.token_index(cu, B, T, is_decode)
    return oracle.row_ids(ids, req, local, ctx, batch.layer_multipliers, batch.vocab_sizes,
                          batch.offsets, batch.ngram_size, batch.heads_per_ngram,
                          batch.boundary_id)


def shard_rows(batch, world, rank):
    """Rank `rank`'s rows of `batch` split `world` ways: the library's plan,
    the shard's inputs from the oracle's carried context, the oracle's hash.
    Returns (token_begin, token_end, rows [L, end - begin, H])."""
    import oracle

    import layer_gram_embedding_gb300 as ple

    cu = batch.cu_seqlens
    tb, te, rb, rc = ple.ple_shard_plan(cu, batch.num_requests, batch.num_tokens, world, rank)
    L, H = batch.num_layers, batch.num_heads
    if te == tb:
        return tb, te, np.zeros((L, 0, H), dtype=np.int64)
    if batch.is_decode:
        return tb, te, _rows(batch.ids[tb:te], None, batch.ngram_context[rb:rb + rc], batch,
                             True)
    # the carried context of every request after the tokens before the cut:
    # the oracle's next-call context of the prefix [0, tb)
    if tb > 0:
        req, local = oracle.token_index(cu, batch.num_requests, batch.num_tokens, False)
        carried = oracle.next_context(batch.ids[:tb], req[:tb], local[:tb], batch.ngram_context)
    else:
        carried = batch.ngram_context
    shard_cu = np.clip(cu[rb:rb + rc + 1].astype(np.int64) - tb, 0, te - tb).astype(np.int32)
    return tb, te, _rows(batch.ids[tb:te], shard_cu, carried[rb:rb + rc], batch, False)


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
            tb, te, mine = shard_rows(full, world, rank)
            gathered = [None] * world
            dist.all_gather_object(gathered, (tb, te, mine))
            if rank == 0:
                gathered.sort(key=lambda g: g[0])
                contiguous = all(a[1] == b[0] for a, b in zip(gathered, gathered[1:]))
                covers = gathered[0][0] == 0 and gathered[-1][1] == full.num_tokens
                whole = np.concatenate([g[2] for g in gathered], axis=1)
                ref = _rows(full.ids, full.cu_seqlens, full.ngram_context, full, full.is_decode)
                results.put((full.name, bool(contiguous and covers and
                                             np.array_equal(whole, ref))))
        worst = d.max(float(rank + 1))
        if rank == 0:
            results.put(("max", worst == float(world)))
        d.barrier()
    finally:
        d.close()


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_shards_equal_the_whole_batch(world):
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = dict(results.get(timeout=10) for _ in range(4))
    assert got == {"ragged_16": True, "mixed_8192": True, "decode_b8": True, "max": True}, got


@pytest.mark.parametrize("world", [1, 2, 7, 64, 40000])
def test_planned_shards_at_any_count_equal_the_whole_batch(world):
    sys.path.insert(0, ROOT)
    import workloads as wl
    full = wl.ragged_16()
    whole = _rows(full.ids, full.cu_seqlens, full.ngram_context, full, False)
    parts = [shard_rows(full, world, r) for r in range(world)]
    assert [p[0] for p in parts] == [full.num_tokens * r // world for r in range(world)]
    assert np.array_equal(np.concatenate([p[2] for p in parts], axis=1), whole)


@pytest.mark.parametrize("cuts", [[0, 1, 29449], [0, 100, 5000, 29449], [0, 29448, 29449]])
def test_slices_at_any_cut_equal_the_whole_batch(cuts):
    sys.path.insert(0, ROOT)
    import workloads as wl
    full = wl.ragged_16()
    whole = _rows(full.ids, full.cu_seqlens, full.ngram_context, full, False)
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        s = wl.slice_batch(full, a, b)
        parts.append(_rows(s.ids, s.cu_seqlens, s.ngram_context, s, False))
    assert np.array_equal(np.concatenate(parts, axis=1), whole)
