"""GPU parity: the CUDA library against the CPU oracle, bit for bit.

Every comparison is array equality: the hash is integer arithmetic, so the
only acceptable difference is none (FreeToken PR #338, "perf(ple): fuse the
n-gram row-id hash into one Triton kernel", section "Why it is safe": the
fused kernel is byte-identical to the reference on prefill and decode shapes
and after CUDA-graph replays).  Inputs come from the seeded generators in
workloads.py; expected values come from the oracle only.
"""

import dataclasses
import os

import numpy as np
import pytest
import torch

import layer_gram_embedding_gb300 as ple
import oracle
import workloads as wl
from brute_force import brute_row_ids

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = torch.device("cuda:0")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def oracle_index(batch):
    return oracle.token_index(batch.cu_seqlens, batch.num_requests, batch.num_tokens,
                              batch.is_decode)


def oracle_rows(batch, req=None, local=None):
    if req is None:
        req, local = oracle_index(batch)
    return oracle.row_ids(batch.ids, req, local, batch.ngram_context, batch.layer_multipliers,
                          batch.vocab_sizes, batch.offsets, batch.ngram_size,
                          batch.heads_per_ngram, batch.boundary_id)


def gpu_index(batch):
    cu = dev(batch.cu_seqlens) if batch.cu_seqlens is not None else None
    return ple.ple_build_token_index(cu, batch.num_requests, batch.num_tokens, batch.is_decode,
                                     device=DEV)


def gpu_rows(batch, ids=None, out=None):
    req, local = gpu_index(batch)
    return ple.ple_row_ids(dev(batch.ids) if ids is None else ids, req, local,
                           dev(batch.ngram_context), dev(batch.layer_multipliers),
                           dev(batch.vocab_sizes), dev(batch.offsets), batch.ngram_size,
                           batch.heads_per_ngram, batch.boundary_id, out=out)


def assert_same(got: torch.Tensor, expect: np.ndarray, what: str):
    g = got.cpu().numpy()
    assert g.shape == expect.shape, what
    if not np.array_equal(g, expect):
        bad = np.argwhere(g != expect)
        raise AssertionError(f"{what}: {len(bad)} of {g.size} differ, first at {bad[0].tolist()}: "
                             f"{g[tuple(bad[0])]} != {expect[tuple(bad[0])]}")


WORKLOADS = {b.name + ("_i32" if b.ids.dtype == np.int32 else ""): b for b in wl.all_workloads()}

# The library hashes a call of at most small_batch_max_rows() row ids with
# the small-batch kernel (one thread per row id) and a larger one with the
# tiled kernels; the edge-case tests run every case through both.
KERNELS = ["small", "tiled"]


def for_kernel(batch, kernel):
    """The batch as it is for the small-batch kernel, or, for the tiled
    kernels, with its layers repeated until the call has more row ids than
    the small-batch kernel takes.  Repeated layers have the same parameters,
    so the oracle's rows repeat with them."""
    limit = ple.small_batch_max_rows()
    rows = batch.row_ids_per_call
    if kernel == "small":
        assert rows <= limit, f"{rows} row ids: more than the small-batch kernel takes"
        return batch
    k = limit // rows + 1
    return dataclasses.replace(batch, layer_multipliers=np.tile(batch.layer_multipliers, (k, 1)),
                               vocab_sizes=np.tile(batch.vocab_sizes, (k, 1)),
                               offsets=np.tile(batch.offsets, (k, 1)))


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_token_index_matches_oracle(name):
    batch = WORKLOADS[name]
    req, local = gpu_index(batch)
    oreq, olocal = oracle_index(batch)
    assert np.array_equal(req.cpu().numpy(), oreq)
    assert np.array_equal(local.cpu().numpy(), olocal)


@pytest.mark.parametrize("decode", [False, True])
def test_token_index_paths(decode):
    """Outputs that are 4- but not 16-byte aligned (scalar stores) and more
    than 4096 requests (cu_seqlens read from global memory)."""
    rng = np.random.default_rng(31)
    B = 5000
    lengths = np.ones(B, np.int64) if decode else rng.integers(0, 4, size=B)
    T = int(lengths.sum())
    cu = wl.cu_from_lengths(lengths)
    oreq, olocal = oracle.token_index(None if decode else cu, B, T, decode)
    buf = torch.full((2, T + 1), -9, dtype=torch.int32, device=DEV)
    req, local = buf[0, 1:], buf[1, 1:]
    assert req.data_ptr() % 16 != 0
    ple.ple_build_token_index(None if decode else dev(cu), B, T, decode, req=req, local=local)
    assert np.array_equal(req.cpu().numpy(), oreq)
    assert np.array_equal(local.cpu().numpy(), olocal)
    assert int(buf[0, 0]) == -9 and int(buf[1, 0]) == -9
    req2, local2 = ple.ple_build_token_index(None if decode else dev(cu), B, T, decode, device=DEV)
    assert np.array_equal(req2.cpu().numpy(), oreq)
    assert np.array_equal(local2.cpu().numpy(), olocal)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_validate_index_accepts_the_built_index(name):
    batch = WORKLOADS[name]
    req, local = gpu_index(batch)
    cu = dev(batch.cu_seqlens) if batch.cu_seqlens is not None else None
    first = ple.ple_validate_index(cu, batch.num_requests, batch.num_tokens, batch.is_decode,
                                   req, local)
    assert int(first) == batch.num_tokens


@pytest.mark.parametrize("decode", [False, True])
def test_validate_index_finds_the_first_wrong_token(decode):
    batch = wl.mixed_8192() if not decode else wl.random_batch(5, decode_batch=True, T_max=5000)
    cu = dev(batch.cu_seqlens) if batch.cu_seqlens is not None else None
    rng = np.random.default_rng(17)
    for trial in range(6):
        req, local = gpu_index(batch)
        T = batch.num_tokens
        picks = rng.choice(T, size=int(rng.integers(1, 5)), replace=False)
        for t in picks:
            if rng.random() < 0.5:
                req[int(t)] += 1
            else:
                local[int(t)] -= 1
        first = ple.ple_validate_index(cu, batch.num_requests, T, batch.is_decode, req, local)
        assert int(first) == int(picks.min())


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_row_ids_match_oracle_full_size(name):
    """Every workload at its full size, in the launch configuration the
    benchmark uses, compared element by element."""
    batch = WORKLOADS[name]
    assert_same(gpu_rows(batch), oracle_rows(batch), name)


def low32(a: np.ndarray) -> np.ndarray:
    """The low 32 bits of int64 values as int32 (two's complement)."""
    return (a.astype(np.uint64) & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.int32)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_int32_row_ids_full_size(name):
    """ple_row_ids_i32: the low 32 bits of every row id."""
    batch = WORKLOADS[name]
    req, local = gpu_index(batch)
    out = ple.ple_row_ids(dev(batch.ids), req, local, dev(batch.ngram_context),
                          dev(batch.layer_multipliers), dev(batch.vocab_sizes), dev(batch.offsets),
                          batch.ngram_size, batch.heads_per_ngram, batch.boundary_id,
                          out_dtype=torch.int32)
    assert out.dtype == torch.int32
    assert_same(out, low32(oracle_rows(batch)), f"{name} int32")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("chunk", range(3))
def test_int32_row_ids_random_edges(chunk, kernel):
    """Random offsets push row ids past 2^31 (the low words wrap); misaligned
    outputs (4- but not 16-byte aligned) take the scalar stores."""
    for seed in range(chunk * 40, (chunk + 1) * 40):
        batch = for_kernel(wl.random_batch(9000 + seed, T_max=150,
                                           ids_dtype=np.int32 if seed % 2 else np.int64,
                                           N=[3, 4, 5, 3, 6][seed % 5],
                                           hpn=[2, 4, 8, 4, 3][seed % 5]), kernel)
        req, local = gpu_index(batch)
        L, T, H = batch.num_layers, batch.num_tokens, batch.num_heads
        buf = torch.full((L * T * H + 1,), 77, dtype=torch.int32, device=DEV)
        out = buf[1:].view(L, T, H) if seed % 3 == 0 else buf[:-1].view(L, T, H)
        ple.ple_row_ids(dev(batch.ids), req, local, dev(batch.ngram_context),
                        dev(batch.layer_multipliers), dev(batch.vocab_sizes), dev(batch.offsets),
                        batch.ngram_size, batch.heads_per_ngram, batch.boundary_id, out=out,
                        out_dtype=torch.int32)
        assert_same(out, low32(oracle_rows(batch)), f"int32 seed {seed}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_int32_row_ids_decode_without_index(kernel):
    batch = for_kernel(wl.decode(8), kernel)
    out = ple.ple_row_ids(dev(batch.ids), None, None, dev(batch.ngram_context),
                          dev(batch.layer_multipliers), dev(batch.vocab_sizes), dev(batch.offsets),
                          3, 2, batch.boundary_id, out_dtype=torch.int32)
    assert_same(out, low32(oracle_rows(batch)), "int32 decode")


def gpu_rows_carry(batch, out_dtype=torch.int64, index_free=False):
    ctx = dev(batch.ngram_context)
    nxt = torch.full_like(ctx, -5)
    if index_free:
        req = local = cu = None
    else:
        req, local = gpu_index(batch)
        cu = dev(batch.cu_seqlens) if batch.cu_seqlens is not None else dev(
            np.arange(batch.num_requests + 1, dtype=np.int32))
    out = ple.ple_row_ids(dev(batch.ids), req, local, ctx, dev(batch.layer_multipliers),
                          dev(batch.vocab_sizes), dev(batch.offsets), batch.ngram_size,
                          batch.heads_per_ngram, batch.boundary_id, out_dtype=out_dtype,
                          cu_seqlens=cu, next_context=nxt)
    return out, nxt


def oracle_carry(batch):
    req, local = oracle_index(batch)
    return oracle.next_context(batch.ids, req, local, batch.ngram_context)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_context_carry_full_size(name):
    """ple_row_ids_ex: the same row ids, plus every request's carried context."""
    batch = WORKLOADS[name]
    out, nxt = gpu_rows_carry(batch)
    assert_same(out, oracle_rows(batch), f"{name} rows with carry")
    assert_same(nxt, oracle_carry(batch), f"{name} carried context")
    if batch.is_decode:
        out, nxt = gpu_rows_carry(batch, index_free=True)
        assert_same(out, oracle_rows(batch), f"{name} rows, index-free carry")
        assert_same(nxt, oracle_carry(batch), f"{name} carried context, index-free")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("chunk", range(3))
def test_context_carry_random_edges(chunk, kernel):
    """Empty requests keep their row, short requests mix context and tokens,
    int32 ids and int32 row ids."""
    for seed in range(chunk * 50, (chunk + 1) * 50):
        batch = for_kernel(wl.random_batch(11000 + seed, T_max=120,
                                           ids_dtype=np.int32 if seed % 2 else np.int64), kernel)
        out_dtype = torch.int32 if seed % 3 == 0 else torch.int64
        out, nxt = gpu_rows_carry(batch, out_dtype=out_dtype)
        exp = oracle_rows(batch)
        assert_same(out, low32(exp) if out_dtype == torch.int32 else exp, f"carry rows {seed}")
        assert_same(nxt, oracle_carry(batch), f"carried context {seed}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_decode_steps_chain_through_the_carry(kernel):
    """Five decode steps, each fed the context the previous step carried,
    against the oracle run step by step."""
    b = for_kernel(wl.decode(8), kernel)
    ctx_o = b.ngram_context.copy()
    ctx_g = dev(b.ngram_context)
    M, vocab, off = dev(b.layer_multipliers), dev(b.vocab_sizes), dev(b.offsets)
    for step in range(5):
        ids = wl.decode(8, 10 + step).ids
        nxt = torch.empty_like(ctx_g)
        out = ple.ple_row_ids(dev(ids), None, None, ctx_g, M, vocab, off, 3, 2, b.boundary_id,
                              next_context=nxt)
        sb = dataclasses.replace(b, ids=ids, ngram_context=ctx_o)
        assert_same(out, oracle_rows(sb), f"decode step {step}")
        ctx_o = oracle_carry(sb)
        assert_same(nxt, ctx_o, f"carry after step {step}")
        ctx_g = nxt


def test_chunked_prefill_through_the_carry_equals_one_prefill():
    """The first request of the large prefill hashed in four chunks, each
    chunk using the context the GPU carried out of the previous one, gives
    the rows of one prefill."""
    full = wl.prefill_262144()
    start = int(full.cu_seqlens[1])  # the first request's length
    first = wl.Batch("r0", full.ids[:start], full.ngram_context[:1],
                     np.array([0, start], np.int32), False, full.layer_multipliers,
                     full.vocab_sizes, full.offsets, 4, 4)
    whole = oracle_rows(first)
    ctx = dev(first.ngram_context)
    cuts = [0, 1, 37, start // 2, start]
    parts = []
    for a, c in zip(cuts[:-1], cuts[1:]):
        chunk = dataclasses.replace(first, ids=first.ids[a:c],
                                    cu_seqlens=np.array([0, c - a], np.int32))
        nxt = torch.empty_like(ctx)
        req, local = ple.ple_build_token_index(dev(chunk.cu_seqlens), 1, c - a, False)
        parts.append(ple.ple_row_ids(dev(chunk.ids), req, local, ctx,
                                     dev(chunk.layer_multipliers), dev(chunk.vocab_sizes),
                                     dev(chunk.offsets), 4, 4, chunk.boundary_id,
                                     cu_seqlens=dev(chunk.cu_seqlens), next_context=nxt))
        ctx = nxt
    got = torch.cat(parts, dim=1)
    assert_same(got, whole, "chunked prefill through the carry")


def check_embed(batch, table, index_free=False, what="", search=False, prepared=False):
    """GPU gather vs the oracle's exact (double) sum: fp32 recursive summation
    of H terms errs by at most (H-1) * 2^-24 * sum|x| per element.  search:
    no index, the requests found from cu_seqlens in the kernel; prepared:
    head constants from ple_prepare_heads."""
    t = torch.from_numpy(table.view(np.int16)).to(DEV)
    cu = None
    if index_free or search:
        req = local = None
        cu = dev(batch_cu(batch)) if search else None
    else:
        req, local = gpu_index(batch)
    heads = (ple.ple_prepare_heads(dev(batch.vocab_sizes), dev(batch.offsets))
             if prepared else None)
    got = ple.ple_row_embed(dev(batch.ids), req, local, dev(batch.ngram_context),
                            dev(batch.layer_multipliers), dev(batch.vocab_sizes),
                            dev(batch.offsets), batch.ngram_size, batch.heads_per_ngram,
                            batch.boundary_id, t, cu_seqlens=cu,
                            heads=heads).cpu().numpy().astype(np.float64)
    oreq, olocal = oracle_index(batch)
    exact, abs_sum = oracle.row_embed(batch.ids, oreq, olocal, batch.ngram_context,
                                      batch.layer_multipliers, batch.vocab_sizes, batch.offsets,
                                      batch.ngram_size, batch.heads_per_ngram, batch.boundary_id,
                                      table)
    bound = (batch.num_heads - 1) * 2.0 ** -24 * abs_sum
    err = np.abs(got - exact)
    assert got.shape == exact.shape
    assert np.all(err <= bound), (what, float(err.max()), float((err - bound).max()))


@pytest.mark.parametrize("D", [8, 16, 24, 64, 256, 264])
def test_row_embed_random_batches(D):
    for seed in range(12):
        batch, table = wl.small_table_batch(12000 + 31 * D + seed, D=D, T_max=150,
                                            ids_dtype=np.int32 if seed % 2 else np.int64)
        # every third batch finds its requests from cu_seqlens in the kernel,
        # every fourth uses prepared head constants
        check_embed(batch, table, what=f"D={D} seed={seed}", search=seed % 3 == 1,
                    prepared=seed % 4 == 2)


def test_row_embed_rows_outside_the_table_add_nothing():
    batch, table = wl.small_table_batch(777, D=32, T_max=200, L=2)
    check_embed(batch, np.ascontiguousarray(table[:, : table.shape[1] // 3]), what="short table")


def test_row_embed_decode_without_an_index():
    b = wl.decode(8)
    rng = np.random.default_rng(8)
    vocab = wl.random_primes(rng, 4, 2, 3000).reshape(1, 4)
    b = dataclasses.replace(b, vocab_sizes=vocab, offsets=wl.prefix_offsets(vocab))
    table = wl.embed_table(rng, 1, int(vocab.sum()), 128)
    check_embed(b, table, index_free=True, what="decode")
    check_embed(b, table, index_free=False, what="decode with index")


def test_row_embed_large_prefill_sample():
    """The large-prefill shape (N=4, 12 heads, 8 layers, int64 ids) on the
    first 20000 tokens, D=64, with a table cut to 2^16 rows per layer so that
    most row ids fall outside it (the out-of-range rule at scale)."""
    full = wl.prefill_262144()
    batch = wl.slice_batch(full, 0, 20000)
    rng = np.random.default_rng(3)
    check_embed(batch, wl.embed_table(rng, 8, 2 ** 16, 64), what="prefill sample")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("chunk", range(6))
def test_random_edge_batches(chunk, kernel):
    """Small ragged batches spanning several 64-token tiles with ragged tails,
    empty requests, decodes, ngram_size 2..8, heads 1..3 per order, 1..3
    layers, boundary densities 0..1, INT64_MIN/MAX multipliers, and vocab
    sizes at the 32-bit edges, negative, tiny and huge."""
    for seed in range(chunk * 60, (chunk + 1) * 60):
        dtype = np.int32 if seed % 3 == 0 else np.int64
        batch = for_kernel(wl.random_batch(seed, T_max=200, ids_dtype=dtype), kernel)
        assert_same(gpu_rows(batch), oracle_rows(batch), f"seed {seed}")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("N,hpn", [(3, 2), (3, 4), (4, 4), (5, 8)])
def test_fixed_shapes_random_edges(N, hpn, kernel):
    """The tuned shapes with ragged tiles, empty requests, boundary densities
    0..1 and every kind of vocab size (so both the 32-bit fast path and the
    general path, whose staging the 32-head shape splits), int64 row ids,
    reading an index and finding the requests from cu_seqlens."""
    for seed in range(30):
        dtype = np.int32 if seed % 2 else np.int64
        batch = for_kernel(wl.random_batch(15000 + 100 * N + 10 * hpn + seed, N=N, hpn=hpn,
                                           T_max=200, ids_dtype=dtype,
                                           vocab_mode="primes" if seed % 3 == 0 else "mixed"),
                           kernel)
        exp = oracle_rows(batch)
        assert_same(gpu_rows(batch), exp, f"N={N} hpn={hpn} seed {seed}")
        # the same batch with the requests found from cu_seqlens in the kernel
        # (the 32-head shape then takes 32-token tiles), with the carry
        out, nxt = gpu_rows_search(batch, carry=True, prepared=seed % 4 == 3)
        assert_same(out, exp, f"N={N} hpn={hpn} seed {seed} search mode")
        assert_same(nxt, oracle_carry(batch), f"N={N} hpn={hpn} seed {seed} search carry")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("N", list(range(9, 17)))
def test_long_ngrams_generic_path(N, kernel):
    batch = for_kernel(wl.random_batch(5000 + N, N=N, hpn=2, L=2, T_max=150), kernel)
    assert_same(gpu_rows(batch), oracle_rows(batch), f"N={N}")


@pytest.mark.parametrize("N,hpn", [(2, 1), (2, 255), (3, 128), (5, 64), (16, 17), (4, 85),
                                   (3, 33), (9, 5)])
@pytest.mark.parametrize("kernel", KERNELS)
def test_head_counts(N, hpn, kernel):
    if (N - 1) * hpn > ple.PLE_MAX_HEADS:
        pytest.skip("beyond PLE_MAX_HEADS")
    batch = for_kernel(wl.random_batch(6000 + N * 1000 + hpn, N=N, hpn=hpn, L=2, T_max=100,
                                       vocab_mode="primes"), kernel)
    assert_same(gpu_rows(batch), oracle_rows(batch), f"N={N} hpn={hpn}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_full_range_ids_and_extreme_boundary(kernel):
    rng = np.random.default_rng(77)
    for b in (wl.I64_MIN, wl.I64_MAX, 0, -1):
        batch = wl.random_batch(int(rng.integers(0, 10 ** 6)), T_max=150, boundary=b)
        ids = rng.integers(wl.I64_MIN, wl.I64_MAX, size=batch.num_tokens, dtype=np.int64,
                           endpoint=True)
        ids[rng.random(batch.num_tokens) < 0.2] = b
        batch.ids = ids
        batch = for_kernel(batch, kernel)
        assert_same(gpu_rows(batch), oracle_rows(batch), f"b={b}")


@pytest.mark.parametrize("dtype", [np.int64, np.int32])
def test_misaligned_ids_take_the_scalar_path(dtype):
    """ids that are element-aligned but not 16-byte aligned."""
    batch = wl.prefill_262144(ids_dtype=dtype)
    batch = wl.Batch("mis", batch.ids[:70001], batch.ngram_context, None, False,
                     batch.layer_multipliers, batch.vocab_sizes, batch.offsets, 4, 4)
    batch.cu_seqlens = wl.cu_from_lengths([30000, 0, 40001, 0])
    padded = torch.zeros(batch.num_tokens + 1, dtype=torch.from_numpy(batch.ids).dtype, device=DEV)
    padded[1:] = dev(batch.ids)
    ids = padded[1:]
    assert ids.data_ptr() % 16 != 0
    assert_same(gpu_rows(batch, ids=ids), oracle_rows(batch), "misaligned")


@pytest.mark.parametrize("make", [wl.prefill_512, wl.ragged_16, wl.mixed_8192])
def test_out_not_16_byte_aligned(make):
    """out that is 8-byte but not 16-byte aligned takes the 8-byte readout."""
    batch = make()
    L, T, H = batch.num_layers, batch.num_tokens, batch.num_heads
    buf = torch.full((L * T * H + 1,), -7, dtype=torch.int64, device=DEV)
    out = buf[1:].view(L, T, H)
    assert out.data_ptr() % 16 != 0
    gpu_rows(batch, out=out)
    assert int(buf[0]) == -7
    assert_same(out, oracle_rows(batch), "misaligned out")


def test_empty_batch():
    batch = wl.prefill_512()
    z = torch.empty(0, dtype=torch.int64, device=DEV)
    zi = torch.empty(0, dtype=torch.int32, device=DEV)
    out = ple.ple_row_ids(z, zi, zi, dev(batch.ngram_context), dev(batch.layer_multipliers),
                          dev(batch.vocab_sizes), dev(batch.offsets), 3, 2, batch.boundary_id)
    assert out.shape == (1, 0, 4)


def test_per_layer_calls_with_row_pointers():
    """A per-layer call passes the layer's rows of the parameter arrays and
    L = 1 (invariant: a multi-layer call's slice l equals it)."""
    batch = wl.mixed_8192()
    full = gpu_rows(batch)
    req, local = gpu_index(batch)
    ids, ctx = dev(batch.ids), dev(batch.ngram_context)
    M, vocab, off = dev(batch.layer_multipliers), dev(batch.vocab_sizes), dev(batch.offsets)
    lib = ple.lib()
    out = torch.empty((batch.num_tokens, batch.num_heads), dtype=torch.int64, device=DEV)
    stream = torch.cuda.current_stream(DEV).cuda_stream
    for l in (0, 17, 47):
        st = lib.ple_row_ids(ids.data_ptr(), ple.PLE_I64, batch.num_tokens, req.data_ptr(),
                             local.data_ptr(), ctx.data_ptr(), batch.num_requests, 4,
                             M.data_ptr() + 8 * l * 5, vocab.data_ptr() + 8 * l * 32,
                             off.data_ptr() + 8 * l * 32, 32, 5, 8, 1, batch.boundary_id,
                             out.data_ptr(), stream)
        assert st == ple.PLE_OK
        assert torch.equal(out, full[l])


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("B", [1, 4, 8, 63, 64, 65, 1000])
def test_decode_without_an_index(B, kernel):
    """req = local = NULL: each token its own request at offset 0."""
    batch = wl.decode(min(B, 8)) if B <= 8 else wl.random_batch(7000 + B, decode_batch=True,
                                                                T_max=B, N=3, hpn=2, L=2)
    if B > 8:
        rng = np.random.default_rng(B)
        batch.ids = rng.integers(0, wl.VOCAB, size=B, dtype=np.int64)
        batch.ngram_context = rng.integers(0, wl.VOCAB, size=(B, 2), dtype=np.int64)
        batch.ngram_context[rng.random((B, 2)) < 0.3] = batch.boundary_id
    batch = for_kernel(batch, kernel)
    out = ple.ple_row_ids(dev(batch.ids), None, None, dev(batch.ngram_context),
                          dev(batch.layer_multipliers), dev(batch.vocab_sizes), dev(batch.offsets),
                          batch.ngram_size, batch.heads_per_ngram, batch.boundary_id)
    assert_same(out, oracle_rows(batch), f"index-free decode B={B}")


@pytest.mark.parametrize("prepared", [False, True])
@pytest.mark.parametrize("kernel", KERNELS)
def test_decode_without_an_index_in_a_graph(kernel, prepared):
    """One launch per decode step: capture once, replay with fresh ids
    (with the head constants prepared once before capture, or not)."""
    b0 = for_kernel(wl.decode(8), kernel)
    ids, ctx = dev(b0.ids), dev(b0.ngram_context)
    M, vocab, off = dev(b0.layer_multipliers), dev(b0.vocab_sizes), dev(b0.offsets)
    heads = ple.ple_prepare_heads(vocab, off) if prepared else None
    out = torch.empty((b0.num_layers, 8, 4), dtype=torch.int64, device=DEV)

    def step():
        ple.ple_row_ids(ids, None, None, ctx, M, vocab, off, 3, 2, b0.boundary_id, out=out,
                        heads=heads)

    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream(DEV).wait_stream(s)
    torch.cuda.synchronize(DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for replay in (1, 2, 3):
        fresh = dataclasses.replace(b0, ids=wl.decode(8, replay).ids,
                                    ngram_context=wl.decode(8, replay).ngram_context)
        ids.copy_(dev(fresh.ids))
        ctx.copy_(dev(fresh.ngram_context))
        g.replay()
        torch.cuda.synchronize(DEV)
        assert_same(out, oracle_rows(fresh), f"index-free replay {replay}")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("kind", ["decode_b1", "decode_b4", "decode_b8", "prefill_512"])
def test_cuda_graph_capture_and_three_replays(kind, kernel):
    """Capture the index build and the hash once on fixed buffers; replay
    three times with fresh ids and context, each equal to the oracle."""
    make = (lambda r: wl.decode(int(kind[-1]), r)) if kind.startswith("decode") else wl.prefill_512
    b0 = for_kernel(make(0), kernel)
    ids, ctx = dev(b0.ids), dev(b0.ngram_context)
    M, vocab, off = dev(b0.layer_multipliers), dev(b0.vocab_sizes), dev(b0.offsets)
    cu = dev(b0.cu_seqlens) if b0.cu_seqlens is not None else None
    T, B = b0.num_tokens, b0.num_requests
    req = torch.empty(T, dtype=torch.int32, device=DEV)
    local = torch.empty(T, dtype=torch.int32, device=DEV)
    out = torch.full((b0.num_layers, T, 4), -123, dtype=torch.int64, device=DEV)

    def step():
        ple.ple_build_token_index(cu, B, T, b0.is_decode, req=req, local=local, device=DEV)
        ple.ple_row_ids(ids, req, local, ctx, M, vocab, off, 3, 2, b0.boundary_id, out=out)

    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(s):
        step()  # the documented call before capture
    torch.cuda.current_stream(DEV).wait_stream(s)
    torch.cuda.synchronize(DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for replay in (1, 2, 3):
        fresh = make(replay)
        nb = dataclasses.replace(b0, ids=fresh.ids, ngram_context=fresh.ngram_context)
        ids.copy_(dev(nb.ids))
        ctx.copy_(dev(nb.ngram_context))
        g.replay()
        torch.cuda.synchronize(DEV)
        assert_same(out, oracle_rows(nb), f"{kind} replay {replay}")


@pytest.mark.parametrize("what", ["ctx", "heads"])
def test_refuses_a_geometry_it_cannot_address(what):
    """ValueError, nothing launched, out untouched (a canary is checked)."""
    batch = wl.prefill_512()
    req, local = gpu_index(batch)
    out = torch.full((1, 512, 4), 0x5EED, dtype=torch.int64, device=DEV)
    ctx = dev(batch.ngram_context)
    hpn = 2
    if what == "ctx":
        ctx = torch.zeros((1, 3), dtype=torch.int64, device=DEV)
    else:
        hpn = 1
    with pytest.raises(ValueError):
        ple.ple_row_ids(dev(batch.ids), req, local, ctx, dev(batch.layer_multipliers),
                        dev(batch.vocab_sizes), dev(batch.offsets), 3, hpn, batch.boundary_id,
                        out=out)
    torch.cuda.synchronize(DEV)
    assert bool((out == 0x5EED).all())


@pytest.mark.parametrize("kernel", KERNELS)
def test_out_of_range_index_data_is_clamped_not_read_out_of_bounds(kernel):
    """req outside [0, B) and local outside [0, t] are device data the host
    cannot check; the kernel clamps them (req into [0, B-1], local into
    [0, t]) and stays in bounds.  The rows then follow the page's addressing
    rule on the clamped values, which the brute force evaluates directly
    (on one layer; the tiled case repeats that layer)."""
    one = wl.random_batch(4242, N=4, hpn=2, L=1, T_max=100, decode_batch=False)
    batch = for_kernel(one, kernel)
    T, B = batch.num_tokens, batch.num_requests
    oreq, olocal = oracle_index(batch)
    rng = np.random.default_rng(9)
    req = oreq.copy()
    local = olocal.copy()
    pick = rng.random(T) < 0.3
    req[pick] = rng.choice([-7, B, B + 100, 2 ** 31 - 1], size=int(pick.sum()))
    pick = rng.random(T) < 0.3
    local[pick] = rng.choice([-3, 10 ** 6, 2 ** 31 - 1], size=int(pick.sum()))
    out = ple.ple_row_ids(dev(batch.ids), dev(req), dev(local), dev(batch.ngram_context),
                          dev(batch.layer_multipliers), dev(batch.vocab_sizes),
                          dev(batch.offsets), 4, 2, batch.boundary_id)
    creq = np.clip(req, 0, B - 1)
    clocal = np.minimum(np.maximum(local, 0), np.arange(T))
    exp = np.array(brute_row_ids(one.ids, creq, clocal, one.ngram_context,
                                 one.layer_multipliers, one.vocab_sizes, one.offsets, 4, 2,
                                 one.boundary_id), dtype=np.int64)
    assert_same(out, np.tile(exp, (batch.num_layers, 1, 1)), "clamped index")


def gpu_rows_prepared(batch, out_dtype=torch.int64, carry=False):
    heads = ple.ple_prepare_heads(dev(batch.vocab_sizes), dev(batch.offsets))
    req, local = gpu_index(batch)
    ctx = dev(batch.ngram_context)
    nxt = torch.full_like(ctx, -5) if carry else None
    cu = None
    if carry:
        cu = dev(batch.cu_seqlens) if batch.cu_seqlens is not None else dev(
            np.arange(batch.num_requests + 1, dtype=np.int32))
    out = ple.ple_row_ids(dev(batch.ids), req, local, ctx, dev(batch.layer_multipliers),
                          dev(batch.vocab_sizes), dev(batch.offsets), batch.ngram_size,
                          batch.heads_per_ngram, batch.boundary_id, out_dtype=out_dtype,
                          cu_seqlens=cu, next_context=nxt, heads=heads)
    return out, nxt


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_prepared_heads_full_size(name):
    """Head constants set up once by ple_prepare_heads give the same rows."""
    batch = WORKLOADS[name]
    out, _ = gpu_rows_prepared(batch)
    assert_same(out, oracle_rows(batch), f"{name} prepared heads")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("chunk", range(2))
def test_prepared_heads_random_edges(chunk, kernel):
    """Every kind of head (32-bit fast path, the general path at the 2^31 /
    2^32 edges, negative and zero vocab sizes) through prepared constants,
    with int32 row ids and the context carry in turn."""
    for seed in range(chunk * 40, (chunk + 1) * 40):
        batch = for_kernel(wl.random_batch(13000 + seed, T_max=150,
                                           ids_dtype=np.int32 if seed % 2 else np.int64), kernel)
        out_dtype = torch.int32 if seed % 3 == 0 else torch.int64
        out, nxt = gpu_rows_prepared(batch, out_dtype=out_dtype, carry=seed % 4 == 1)
        exp = oracle_rows(batch)
        assert_same(out, low32(exp) if out_dtype == torch.int32 else exp, f"prepared {seed}")
        if nxt is not None:
            assert_same(nxt, oracle_carry(batch), f"prepared carry {seed}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_prepared_heads_replace_vocab_and_offsets(kernel):
    """With prepared constants the call reads neither vocab_sizes nor
    offsets: NULL for both through the C ABI."""
    batch = for_kernel(wl.random_batch(4711, N=4, hpn=3, L=2, T_max=150), kernel)
    heads = ple.ple_prepare_heads(dev(batch.vocab_sizes), dev(batch.offsets))
    req, local = gpu_index(batch)
    ids, ctx, M = dev(batch.ids), dev(batch.ngram_context), dev(batch.layer_multipliers)
    L, T, H = batch.num_layers, batch.num_tokens, batch.num_heads
    out = torch.full((L, T, H), -1, dtype=torch.int64, device=DEV)
    st = ple.lib().ple_row_ids_ex(ids.data_ptr(), ple.PLE_I64, T, req.data_ptr(),
                                  local.data_ptr(), ctx.data_ptr(), batch.num_requests, 3,
                                  M.data_ptr(), None, None, H, 4, 3, L, batch.boundary_id,
                                  out.data_ptr(), ple.PLE_I64, None, None, heads.data_ptr(),
                                  torch.cuda.current_stream(DEV).cuda_stream)
    assert st == ple.PLE_OK
    assert_same(out, oracle_rows(batch), "prepared heads, no vocab / offsets")


def batch_cu(batch):
    """The batch's cu_seqlens (a decode's is 0, 1, ..., B)."""
    if batch.cu_seqlens is not None:
        return batch.cu_seqlens
    return np.arange(batch.num_requests + 1, dtype=np.int32)


def gpu_rows_search(batch, out_dtype=torch.int64, carry=False, prepared=False, out=None):
    """Row ids with req = local = None and cu_seqlens: the kernel searches
    cu_seqlens for each token's request (no index built or read)."""
    ctx = dev(batch.ngram_context)
    nxt = torch.full_like(ctx, -5) if carry else None
    heads = (ple.ple_prepare_heads(dev(batch.vocab_sizes), dev(batch.offsets))
             if prepared else None)
    got = ple.ple_row_ids(dev(batch.ids), None, None, ctx, dev(batch.layer_multipliers),
                          dev(batch.vocab_sizes), dev(batch.offsets), batch.ngram_size,
                          batch.heads_per_ngram, batch.boundary_id, out=out, out_dtype=out_dtype,
                          cu_seqlens=dev(batch_cu(batch)), next_context=nxt, heads=heads)
    return got, nxt


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_cu_search_mode_full_size(name):
    """Every workload with the index found in the kernel from cu_seqlens:
    the same rows (int64 and int32, derived and prepared constants) and the
    same carried context as the oracle."""
    batch = WORKLOADS[name]
    exp = oracle_rows(batch)
    out, nxt = gpu_rows_search(batch, carry=True)
    assert_same(out, exp, f"{name} search mode")
    assert_same(nxt, oracle_carry(batch), f"{name} search mode carry")
    out, _ = gpu_rows_search(batch, out_dtype=torch.int32, prepared=True)
    assert_same(out, low32(exp), f"{name} search mode, int32, prepared")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("chunk", range(3))
def test_cu_search_mode_random_edges(chunk, kernel):
    """Empty requests (repeated cu_seqlens entries, at the start, the end and
    in runs), one-token requests, decodes given as cu_seqlens, ragged tiles,
    with the carry and int32 row ids in turn."""
    for seed in range(chunk * 50, (chunk + 1) * 50):
        batch = for_kernel(wl.random_batch(17000 + seed, T_max=150,
                                           ids_dtype=np.int32 if seed % 2 else np.int64), kernel)
        out_dtype = torch.int32 if seed % 3 == 0 else torch.int64
        out, nxt = gpu_rows_search(batch, out_dtype=out_dtype, carry=seed % 4 == 1,
                                   prepared=seed % 5 == 2)
        exp = oracle_rows(batch)
        assert_same(out, low32(exp) if out_dtype == torch.int32 else exp, f"search {seed}")
        if nxt is not None:
            assert_same(nxt, oracle_carry(batch), f"search carry {seed}")


@pytest.mark.parametrize("kernel,B", [("small", 1000), ("tiled", 500), ("tiled", 600),
                                      ("tiled", 1000), ("tiled", 3000)])
def test_cu_search_mode_many_requests(kernel, B):
    """Hundreds to thousands of requests, many of them empty or one token
    long, so a tile spans anywhere from one request to dozens: two rounds
    of the warp's 32-way search (B = 500, 600, 1000) or three (B = 3000)."""
    rng = np.random.default_rng(4321 + B)
    lengths = rng.choice([0, 1, 1, 2, 5, 40], size=B)
    if B in (500, 600):
        lengths = rng.choice([0, 1, 2, 40, 100], size=B)
    T = int(lengths.sum())
    base = wl.random_batch(99, N=4, hpn=4, L=4 if B in (500, 600) else 1, T_max=10,
                           decode_batch=False)
    batch = dataclasses.replace(
        base, ids=rng.integers(0, wl.VOCAB, size=T, dtype=np.int64),
        ngram_context=rng.integers(0, wl.VOCAB, size=(B, 3), dtype=np.int64),
        cu_seqlens=wl.cu_from_lengths(lengths))
    batch = for_kernel(batch, kernel)
    out, nxt = gpu_rows_search(batch, carry=True)
    assert_same(out, oracle_rows(batch), "many requests")
    assert_same(nxt, oracle_carry(batch), "many requests carry")


def test_cu_search_mode_in_a_graph():
    """A prefill step of one launch (no index build) captured once and
    replayed with fresh ids and contexts."""
    b0 = wl.ragged_16()
    ids, ctx = dev(b0.ids), dev(b0.ngram_context)
    M, vocab, off = dev(b0.layer_multipliers), dev(b0.vocab_sizes), dev(b0.offsets)
    cu = dev(b0.cu_seqlens)
    out = torch.full((1, b0.num_tokens, b0.num_heads), -1, dtype=torch.int64, device=DEV)

    def step():
        ple.ple_row_ids(ids, None, None, ctx, M, vocab, off, b0.ngram_size, b0.heads_per_ngram,
                        b0.boundary_id, out=out, cu_seqlens=cu)

    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream(DEV).wait_stream(s)
    torch.cuda.synchronize(DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for replay in (1, 2, 3):
        rng = np.random.default_rng(600 + replay)
        fresh_ids = wl.uniform_ids(rng, b0.num_tokens, 0.02)
        fresh_ctx = wl.uniform_ids(rng, b0.num_requests * 2, 0.02).reshape(-1, 2)
        nb = dataclasses.replace(b0, ids=fresh_ids, ngram_context=fresh_ctx)
        ids.copy_(dev(nb.ids))
        ctx.copy_(dev(nb.ngram_context))
        g.replay()
        torch.cuda.synchronize(DEV)
        assert_same(out, oracle_rows(nb), f"search-mode replay {replay}")


@pytest.mark.parametrize("hpn", [2, 4])
@pytest.mark.parametrize("kernel", KERNELS)
def test_cu_search_mode_malformed_cu_stays_in_bounds(kernel, hpn):
    """cu_seqlens is device data the host cannot check.  Malformed contents
    (negative, past T, decreasing) give unspecified rows but no access
    outside the arrays: the canaries around the output and the carried
    context survive, and the call completes.  hpn = 4 is a fixed shape (the
    warp search and lane ranking of the fixed-shape kernel), hpn = 2 a
    runtime one (a per-lane search)."""
    batch = for_kernel(wl.random_batch(5150, N=4, hpn=hpn, L=1, T_max=100, decode_batch=False),
                       kernel)
    L, T, H, B = batch.num_layers, batch.num_tokens, batch.num_heads, batch.num_requests
    rng = np.random.default_rng(3)
    cu = rng.choice([-(2 ** 31), -5, 0, 3, T, T + 7, 2 ** 31 - 1], size=B + 1).astype(np.int32)
    buf = torch.full((L * T * H + 2,), 0x5A5A, dtype=torch.int64, device=DEV)
    out = buf[1:-1].view(L, T, H)
    ctx = dev(batch.ngram_context)
    nbuf = torch.full((B * 3 + 2,), 77, dtype=torch.int64, device=DEV)
    nxt = nbuf[1:-1].view(B, 3)
    ple.ple_row_ids(dev(batch.ids), None, None, ctx, dev(batch.layer_multipliers),
                    dev(batch.vocab_sizes), dev(batch.offsets), 4, hpn, batch.boundary_id, out=out,
                    cu_seqlens=dev(cu), next_context=nxt)
    torch.cuda.synchronize(DEV)
    assert int(buf[0]) == 0x5A5A and int(buf[-1]) == 0x5A5A
    assert int(nbuf[0]) == 77 and int(nbuf[-1]) == 77


@pytest.mark.parametrize("extra", [0, 1])
def test_small_and_tiled_kernels_meet_at_the_threshold(extra):
    """The large prefill's first tokens, as many as the small-batch kernel
    takes (96 row ids per token) and one token more (the tiled kernels)."""
    full = wl.prefill_262144()
    per_token = full.num_layers * full.num_heads
    T = ple.small_batch_max_rows() // per_token + extra
    batch = wl.slice_batch(full, 0, T)
    assert (batch.row_ids_per_call <= ple.small_batch_max_rows()) == (extra == 0)
    assert_same(gpu_rows(batch), oracle_rows(batch), f"T={T}")


def test_floor_mod_routine_matches_cuda_remainder():
    """The invariant-divisor floored remainder against CUDA's own % plus the
    sign fix, and against Python's floored %, on edge values."""
    xs = [0, 1, -1, 2, -2, 10, -10, wl.I64_MAX, wl.I64_MIN, wl.I64_MIN + 1, wl.I64_MAX - 1,
          2 ** 31, -(2 ** 31), 2 ** 32 - 1, -(2 ** 32), 2 ** 62, -(2 ** 62), 3 * 2 ** 61]
    vs = wl.EDGE_VOCABS + [0, 5, 6, 2 ** 31 - 2, 2 ** 33 + 1, 2 ** 63 - 25]
    pairs = [(x, v) for x in xs for v in vs]
    for v in vs:
        if v not in (0,):
            for k in (-3, -2, -1, 1, 2, 3):
                for d in (-1, 0, 1):
                    y = k * v + d
                    if wl.I64_MIN <= y <= wl.I64_MAX:
                        pairs.append((y, v))
    rng = np.random.default_rng(1)
    rx = rng.integers(wl.I64_MIN, wl.I64_MAX, size=200000, dtype=np.int64, endpoint=True)
    rv = rng.integers(wl.I64_MIN, wl.I64_MAX, size=200000, dtype=np.int64, endpoint=True)
    rv = rv >> rng.integers(0, 63, size=200000)
    x = np.concatenate([np.array([p[0] for p in pairs], np.int64), rx])
    v = np.concatenate([np.array([p[1] for p in pairs], np.int64), rv])
    fast, ref = ple.ple_selftest_floor_mod(dev(x), dev(v))
    fast, ref = fast.cpu().numpy(), ref.cpu().numpy()
    assert np.array_equal(fast, ref)
    expect = np.array([(int(a) % int(b)) if b != 0 else 0 for a, b in zip(x, v)], dtype=np.int64)
    assert np.array_equal(fast, expect)


def test_floor_mod_fast_path_divisor_sweep():
    """The 32-bit fast path (0 < v <= 2^29) over every divisor up to 2^16 and
    20000 random ones up to 2^29 (plus the powers of two and their
    neighbours, and the first divisors past 2^29, which take the general
    path), each with dividends at the ends of the int64 range, at multiples
    of v +- 1 near them, and with the offset-binary low word all ones (the
    quotient estimate's dropped carries are largest there).  Expected values
    from numpy's floored remainder, which takes the divisor's sign."""
    rng = np.random.default_rng(7)
    vs = np.concatenate([
        np.arange(1, 2 ** 16 + 1, dtype=np.int64),
        rng.integers(2 ** 16, 2 ** 29, size=20000, endpoint=True, dtype=np.int64),
        np.array([2 ** k + d for k in range(1, 30) for d in (-1, 0, 1)] + [2 ** 29 + 2, 2 ** 30],
                 dtype=np.int64)])
    vs = vs[vs > 0]
    lo_ones = np.int64(0xFFFFFFFF)
    per_v = []
    big = wl.I64_MAX // vs  # multiples of v near the ends
    per_v.append(np.full_like(vs, wl.I64_MIN))
    per_v.append(np.full_like(vs, wl.I64_MAX))
    per_v.append(np.full_like(vs, -1))
    per_v.append(np.zeros_like(vs))
    for d in (-1, 0, 1):
        per_v.append(big * vs + d if d <= 0 else big * vs - vs + d)
        per_v.append(-big * vs + d)
    hi = rng.integers(-(2 ** 31), 2 ** 31, size=vs.size, dtype=np.int64)
    per_v.append((hi << 32) | lo_ones)          # low word all ones (offset binary too)
    per_v.append((hi << 32) | lo_ones ^ (1 << 31))
    per_v.append(rng.integers(wl.I64_MIN, wl.I64_MAX, size=vs.size, endpoint=True,
                              dtype=np.int64))
    x = np.concatenate(per_v)
    v = np.tile(vs, len(per_v))
    fast, ref = ple.ple_selftest_floor_mod(dev(x), dev(v))
    fast = fast.cpu().numpy()
    assert np.array_equal(fast, ref.cpu().numpy())
    assert np.array_equal(fast, np.remainder(x, v))


def test_stream_argument_is_honoured():
    batch = wl.ragged_16()
    s = torch.cuda.Stream(DEV)
    with torch.cuda.stream(s):
        out = gpu_rows(batch)
    s.synchronize()
    assert_same(out, oracle_rows(batch), "side stream")


def test_binding_refuses_malformed_new_arguments():
    """The binding's checks on the prepared constants and cu_seqlens: wrong
    shape, dtype or length is a ValueError / TypeError before any launch."""
    b = wl.prefill_512()
    ids, ctx = dev(b.ids), dev(b.ngram_context)
    M, vocab, off = dev(b.layer_multipliers), dev(b.vocab_sizes), dev(b.offsets)
    heads = ple.ple_prepare_heads(vocab, off)
    assert tuple(heads.shape) == (1, 4, ple.PLE_HEAD_BYTES) and heads.dtype == torch.uint8
    args = (ids, None, None, ctx, M, vocab, off, 3, 2, b.boundary_id)
    with pytest.raises(ValueError):
        ple.ple_row_ids(*args, heads=heads[:, :3])  # wrong number of heads
    with pytest.raises(TypeError):
        ple.ple_row_ids(*args, heads=heads.view(torch.int8))  # not uint8
    with pytest.raises(ValueError):
        ple.ple_row_ids(*args, cu_seqlens=dev(np.array([0, 256, 512], np.int32)))  # B + 1 != 2
    with pytest.raises(TypeError):
        ple.ple_row_ids(*args, cu_seqlens=dev(np.array([0, 512], np.int64)))  # not int32
    with pytest.raises(ValueError):
        ple.ple_prepare_heads(vocab, off[:, :3])  # shapes differ
    with pytest.raises(ValueError):
        req, _ = gpu_index(b)
        ple.ple_row_ids(ids, req, None, ctx, M, vocab, off, 3, 2, b.boundary_id)  # one of two
    # and the well-formed calls agree
    exp = oracle_rows(b)
    assert_same(ple.ple_row_ids(*args, heads=heads, cu_seqlens=dev(b.cu_seqlens)), exp,
                "well-formed search mode with prepared constants")


FUZZ_SHAPES = [(3, 2), (3, 4), (4, 4), (5, 8)]
FUZZ_MODES = ["arrays", "arrays_i32", "search", "carry", "prepared", "index_free", "misaligned"]


def fuzz_case(seed):
    """One random call: the kernel (small-batch or tiled), the shape (a tuned
    fixed shape 60% of the time, else random), the ids dtype, the vocab mix,
    the way the index is given, the output dtype, the context carry and
    prepared constants all drawn from the seed."""
    rng = np.random.default_rng(seed)
    kernel = "small" if seed % 2 else "tiled"
    N, hpn = FUZZ_SHAPES[rng.integers(0, 4)] if rng.random() < 0.6 else (None, None)
    b = wl.random_batch(seed, T_max=int(rng.choice([8, 64, 150, 400])), N=N, hpn=hpn,
                        ids_dtype=np.int32 if rng.random() < 0.4 else np.int64,
                        vocab_mode="primes" if rng.random() < 0.5 else "mixed")
    if kernel == "small" and b.row_ids_per_call > ple.small_batch_max_rows():
        kernel = "tiled"
    b = for_kernel(b, kernel)
    mode = str(rng.choice(FUZZ_MODES))
    if mode == "index_free" and not b.is_decode:
        mode = "search"
    out_dtype = torch.int32 if rng.random() < 0.4 else torch.int64
    carry, prepared = bool(rng.random() < 0.5), bool(rng.random() < 0.5)
    nxt = None
    if mode in ("arrays", "misaligned"):
        out_dtype = torch.int64
        out = None
        if mode == "misaligned":
            L, T, H = b.num_layers, b.num_tokens, b.num_heads
            out = torch.full((L * T * H + 1,), 7, dtype=torch.int64, device=DEV)[1:].view(L, T, H)
        got = gpu_rows(b, out=out)
    elif mode == "arrays_i32":
        out_dtype = torch.int32
        req, local = gpu_index(b)
        got = ple.ple_row_ids(dev(b.ids), req, local, dev(b.ngram_context),
                              dev(b.layer_multipliers), dev(b.vocab_sizes), dev(b.offsets),
                              b.ngram_size, b.heads_per_ngram, b.boundary_id, out_dtype=out_dtype)
    elif mode == "search":
        got, nxt = gpu_rows_search(b, out_dtype=out_dtype, carry=carry, prepared=prepared)
    elif mode == "carry":
        got, nxt = gpu_rows_carry(b, out_dtype=out_dtype)
    elif mode == "prepared":
        got, nxt = gpu_rows_prepared(b, out_dtype=out_dtype, carry=carry)
    else:
        got, nxt = gpu_rows_carry(b, out_dtype=out_dtype, index_free=True)
    exp = oracle_rows(b)
    what = f"fuzz seed {seed} ({kernel}, {mode})"
    assert_same(got, low32(exp) if out_dtype == torch.int32 else exp, what)
    if nxt is not None:
        assert_same(nxt, oracle_carry(b), what + " carry")


def test_random_call_fuzz():
    """Random calls across every entry-point variant, each against the
    oracle.  PLE_FUZZ_BATCHES sets how many (default 1500, a few seconds)
    and PLE_FUZZ_SEED the first seed (default 200000); seeds are
    consecutive, so a failure names its seed."""
    count = int(os.environ.get("PLE_FUZZ_BATCHES", "1500"))
    first = int(os.environ.get("PLE_FUZZ_SEED", "200000"))
    for seed in range(first, first + count):
        fuzz_case(seed)
