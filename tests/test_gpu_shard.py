"""GPU: a batch split across ranks by token range (ple_shard_plan on the host,
ple_shard_inputs on the device) hashes to the same rows as the whole batch.

Each rank's share is hashed as a batch of its own, one rank after another on
one GPU (the ranks never wait on each other: there is no exchange).  The
shard's cu_seqlens and context rows are compared with their definition --
cu_seqlens rebased to the cut and clamped, and each request's carried
context after the tokens before the cut, from the oracle's next-call context
-- and the shard's row ids with rows token_begin..token_end-1 of the whole
batch from the oracle, by array equality."""

import numpy as np
import pytest
import torch

import layer_gram_embedding_gb300 as ple
import oracle
import workloads as wl

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = torch.device("cuda:0")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def whole_rows(batch):
    req, local = oracle.token_index(batch.cu_seqlens, batch.num_requests, batch.num_tokens, False)
    rows = oracle.row_ids(batch.ids, req, local, batch.ngram_context, batch.layer_multipliers,
                          batch.vocab_sizes, batch.offsets, batch.ngram_size,
                          batch.heads_per_ngram, batch.boundary_id)
    return rows, req, local


def expected_shard(batch, req, local, plan):
    tb, te, rb, rc = plan
    cu = batch.cu_seqlens.astype(np.int64)
    shard_cu = np.clip(cu[rb:rb + rc + 1] - tb, 0, te - tb).astype(np.int32)
    if tb > 0:
        carried = oracle.next_context(batch.ids[:tb], req[:tb], local[:tb], batch.ngram_context)
    else:
        carried = batch.ngram_context
    return shard_cu, carried[rb:rb + rc]


def check_split(batch, world, rows=None):
    rows_req_local = whole_rows(batch) if rows is None else rows
    rows, req, local = rows_req_local
    ids, cu, ctx = dev(batch.ids), dev(batch.cu_seqlens), dev(batch.ngram_context)
    M, vocab, off = (dev(batch.layer_multipliers), dev(batch.vocab_sizes), dev(batch.offsets))
    for k in range(world):
        plan = ple.ple_shard_plan(batch.cu_seqlens, batch.num_requests, batch.num_tokens, world,
                                  k)
        tb, te, rb, rc = plan
        if te == tb:
            continue
        s_ids, s_cu, s_ctx = ple.ple_shard_inputs(ids, cu, ctx, plan)
        e_cu, e_ctx = expected_shard(batch, req, local, plan)
        torch.cuda.synchronize()
        assert np.array_equal(s_cu.cpu().numpy(), e_cu), (batch.name, world, k)
        assert np.array_equal(s_ctx.cpu().numpy(), e_ctx), (batch.name, world, k)
        got = ple.ple_row_ids(s_ids, None, None, s_ctx, M, vocab, off, batch.ngram_size,
                              batch.heads_per_ngram, batch.boundary_id, cu_seqlens=s_cu)
        g = got.cpu().numpy()
        if not np.array_equal(g, rows[:, tb:te, :]):
            bad = int((g != rows[:, tb:te, :]).sum())
            raise AssertionError(f"{batch.name} world {world} rank {k}: {bad} row ids differ")


@pytest.mark.parametrize("name", ["prefill_512", "ragged_16", "mixed_8192", "prefill_262144",
                                  "prefill_262144_i32"])
def test_shards_equal_the_whole_batch(name):
    if name == "prefill_262144_i32":
        batch = wl.prefill_262144(ids_dtype=np.int32)
    else:
        batch = {"prefill_512": wl.prefill_512, "ragged_16": wl.ragged_16,
                 "mixed_8192": wl.mixed_8192, "prefill_262144": wl.prefill_262144}[name]()
    rows = whole_rows(batch)
    for world in (2, 3, 8):
        check_split(batch, world, rows)


@pytest.mark.parametrize("seed", range(12))
def test_shards_of_random_batches_with_empty_requests(seed):
    batch = wl.random_batch(500 + seed, T_max=200, decode_batch=False,
                            ids_dtype=np.int32 if seed % 3 == 0 else np.int64)
    rows = whole_rows(batch)
    for world in (1, 2, 5, batch.num_tokens, batch.num_tokens + 3):
        check_split(batch, world, rows)


def test_malformed_device_cu_seqlens_stays_in_bounds():
    """cu_seqlens on the device that disagree with the host's plan give
    unspecified shard inputs, never an access outside the arrays: canaries
    around the outputs stay intact."""
    batch = wl.ragged_16()
    rng = np.random.default_rng(7)
    for trial in range(4):
        bad = rng.integers(-10 ** 6, 10 ** 6, size=batch.cu_seqlens.shape[0]).astype(np.int32)
        plan = ple.ple_shard_plan(batch.cu_seqlens, batch.num_requests, batch.num_tokens, 3,
                                  trial % 3)
        tb, te, rb, rc = plan
        C = batch.ngram_size - 1
        cu_buf = torch.full((rc + 3,), -7, dtype=torch.int32, device=DEV)
        ctx_buf = torch.full((rc + 2, C), -7, dtype=torch.int64, device=DEV)
        ple.ple_shard_inputs(dev(batch.ids), dev(bad), dev(batch.ngram_context), plan,
                             shard_cu_seqlens=cu_buf[1:rc + 2], shard_context=ctx_buf[1:rc + 1])
        torch.cuda.synchronize()
        assert int(cu_buf[0]) == -7 and int(cu_buf[-1]) == -7
        assert (ctx_buf[0] == -7).all() and (ctx_buf[-1] == -7).all()
        s_cu = cu_buf[1:rc + 2].cpu().numpy()
        assert ((s_cu >= 0) & (s_cu <= te - tb)).all()


def test_shard_step_in_a_cuda_graph_with_fresh_inputs():
    """ple_shard_inputs + the one-launch row-id call captured once, replayed
    three times with fresh ids and context copied into the captured inputs:
    each replay equals the oracle's rows of that batch's share."""
    base = wl.prefill_262144()
    world, rank = 3, 1
    plan = ple.ple_shard_plan(base.cu_seqlens, base.num_requests, base.num_tokens, world, rank)
    tb, te, rb, rc = plan
    ids = dev(base.ids)
    ctx = dev(base.ngram_context)
    cu = dev(base.cu_seqlens)
    M, vocab, off = (dev(base.layer_multipliers), dev(base.vocab_sizes), dev(base.offsets))
    s_cu = torch.empty(rc + 1, dtype=torch.int32, device=DEV)
    s_ctx = torch.empty((rc, base.ngram_size - 1), dtype=torch.int64, device=DEV)
    out = torch.empty((base.num_layers, te - tb, base.num_heads), dtype=torch.int64, device=DEV)

    def step():
        s_ids, _, _ = ple.ple_shard_inputs(ids, cu, ctx, plan, shard_cu_seqlens=s_cu,
                                           shard_context=s_ctx)
        ple.ple_row_ids(s_ids, None, None, s_ctx, M, vocab, off, base.ngram_size,
                        base.heads_per_ngram, base.boundary_id, out=out, cu_seqlens=s_cu)

    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream(DEV).wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for replay in range(1, 4):
        fresh = wl.prefill_262144(replay=replay)
        # the same request layout (the plan is fixed at capture): fresh ids and context
        ids_np = fresh.ids.copy()
        ids_np[base.cu_seqlens[:-1]] = base.boundary_id
        ids.copy_(torch.from_numpy(ids_np))
        ctx.copy_(torch.from_numpy(fresh.ngram_context))
        g.replay()
        torch.cuda.synchronize()
        b = wl.replace(base, ids=ids_np, ngram_context=fresh.ngram_context)
        rows, _, _ = whole_rows(b)
        assert np.array_equal(out.cpu().numpy(), rows[:, tb:te, :]), replay


def test_calls_without_programmatic_launch_give_the_same_rows():
    """ple_set_programmatic_launch(False) changes how kernels are launched,
    not what they compute."""
    batch = wl.ragged_16()
    rows, _, _ = whole_rows(batch)
    args = (dev(batch.ids), None, None, dev(batch.ngram_context), dev(batch.layer_multipliers),
            dev(batch.vocab_sizes), dev(batch.offsets), batch.ngram_size, batch.heads_per_ngram,
            batch.boundary_id)
    prev = ple.set_programmatic_launch(False)
    try:
        got = [ple.ple_row_ids(*args, cu_seqlens=dev(batch.cu_seqlens)) for _ in range(3)]
        req, local = ple.ple_build_token_index(dev(batch.cu_seqlens), batch.num_requests,
                                               batch.num_tokens, False)
        got.append(ple.ple_row_ids(dev(batch.ids), req, local, *args[3:]))
    finally:
        ple.set_programmatic_launch(prev)
    torch.cuda.synchronize()
    for g in got:
        assert np.array_equal(g.cpu().numpy(), rows)


def test_binding_refuses_inputs_that_do_not_fit_the_plan():
    batch = wl.ragged_16()
    ids, cu, ctx = dev(batch.ids), dev(batch.cu_seqlens), dev(batch.ngram_context)
    plan = ple.ple_shard_plan(batch.cu_seqlens, batch.num_requests, batch.num_tokens, 2, 1)
    with pytest.raises(ValueError):
        ple.ple_shard_inputs(ids, cu[:-1], ctx, plan)          # cu_seqlens one short
    with pytest.raises(ValueError):
        ple.ple_shard_inputs(ids[:10], cu, ctx, plan)          # fewer ids than the plan's tokens
    tb, te, rb, rc = plan
    with pytest.raises(ValueError):
        ple.ple_shard_inputs(ids, cu, ctx, (tb, te, rb, batch.num_requests))  # past the last request
    with pytest.raises(ValueError):
        ple.ple_shard_inputs(ids, cu, ctx, (tb, tb, rb, 0))    # an empty share
