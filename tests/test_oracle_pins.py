"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test ties the oracle to a hand-worked window, a pure-Python brute force
that addresses tokens without the packed window, a textbook definition, or an
invariant that the definition in FreeToken PR #338 ("perf(ple): fuse the
n-gram row-id hash into one Triton kernel", sections "What" and "Why it is
safe") implies.
"""

import json
import os

import numpy as np
import pytest

import oracle
import workloads as wl
from brute_force import brute_row_ids

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")
I64_MIN, I64_MAX = -(2 ** 63), 2 ** 63 - 1


def run_oracle(batch: wl.Batch, reading="A"):
    req, local = oracle.token_index(batch.cu_seqlens, batch.num_requests, batch.num_tokens,
                                    batch.is_decode)
    return oracle.row_ids(batch.ids, req, local, batch.ngram_context, batch.layer_multipliers,
                          batch.vocab_sizes, batch.offsets, batch.ngram_size,
                          batch.heads_per_ngram, batch.boundary_id, reading)


def run_brute(batch: wl.Batch, reading="A"):
    req, local = oracle.token_index(batch.cu_seqlens, batch.num_requests, batch.num_tokens,
                                    batch.is_decode)
    return np.array(brute_row_ids(batch.ids, req, local, batch.ngram_context,
                                  batch.layer_multipliers, batch.vocab_sizes, batch.offsets,
                                  batch.ngram_size, batch.heads_per_ngram, batch.boundary_id,
                                  reading), dtype=np.int64).reshape(batch.num_layers,
                                                                    batch.num_tokens,
                                                                    batch.num_heads)


def golden_batch(d, name="golden"):
    return wl.Batch(name, np.array(d["input_ids"], np.int64), np.array(d["ngram_context"], np.int64),
                    np.array(d["cu_seqlens"], np.int32), False,
                    np.array(d["layer_multipliers"], np.int64), np.array(d["vocab_sizes"], np.int64),
                    np.array(d["offsets"], np.int64), d["ngram_size"], d["heads_per_ngram"],
                    d["boundary_id"])


# --------------------------------------------------------------------------
# hand-worked values


def test_worked_example_reading_a_and_b():
    g = json.load(open(GOLDEN))
    batch = golden_batch(g["setup"])
    assert run_oracle(batch, "A").tolist() == g["expected_reading_a"]
    assert run_oracle(batch, "B").tolist() == g["expected_reading_b"]
    assert run_brute(batch, "A").tolist() == g["expected_reading_a"]
    assert run_brute(batch, "B").tolist() == g["expected_reading_b"]


@pytest.mark.parametrize("i", [0, 1])
def test_sign_and_wrap_pins(i):
    d = json.load(open(GOLDEN))["sign_and_wrap"][i]
    batch = golden_batch(d)
    assert run_oracle(batch).tolist() == d["expected"]
    assert run_brute(batch).tolist() == d["expected"]


# --------------------------------------------------------------------------
# floored remainder against Python's own floored %


EDGE_X = [0, 1, -1, 2, -2, 10, -10, 11, -11, 12, -12, I64_MAX, I64_MIN, I64_MIN + 1, I64_MAX - 1,
          2 ** 31, -(2 ** 31), 2 ** 32, -(2 ** 32), 2 ** 62, -(2 ** 62), 123456789123, -987654321987]


@pytest.mark.parametrize("v", [v for v in wl.EDGE_VOCABS])
def test_floor_mod_matches_python(v):
    for x in EDGE_X + [v, -v if v != I64_MIN else v, v - 1, v + 1, 2 * v, 3 * v - 1]:
        if not (I64_MIN <= x <= I64_MAX):
            continue
        assert oracle.floor_mod(x, v) == x % v, (x, v)


def test_floor_mod_random():
    rng = np.random.default_rng(7)
    xs = rng.integers(I64_MIN, I64_MAX, size=3000, dtype=np.int64, endpoint=True)
    vs = rng.integers(I64_MIN, I64_MAX, size=3000, dtype=np.int64, endpoint=True)
    vs = np.where(rng.random(3000) < 0.5, vs >> rng.integers(0, 63, size=3000), vs)
    for x, v in zip(xs.tolist(), vs.tolist()):
        if v == 0:
            continue
        assert oracle.floor_mod(x, v) == x % v


# --------------------------------------------------------------------------
# token index against a numpy searchsorted definition


def test_token_index_prefill_matches_searchsorted():
    rng = np.random.default_rng(11)
    for _ in range(200):
        B = int(rng.integers(1, 20))
        lengths = rng.integers(0, 30, size=B)
        cu = wl.cu_from_lengths(lengths)
        T = int(cu[-1])
        req, local = oracle.token_index(cu, B, T, False)
        t = np.arange(T)
        r_ref = np.searchsorted(cu, t, side="right") - 1
        assert np.array_equal(req, r_ref)
        assert np.array_equal(local, t - cu[r_ref])


def test_token_index_decode_vs_one_request_prefill():
    # a decode of B requests and a prefill of one B-token request have the
    # same [T] and opposite meaning ("Why it is safe", the index memo note)
    B = 6
    rq, lq = oracle.token_index(None, B, B, True)
    assert rq.tolist() == list(range(B)) and lq.tolist() == [0] * B
    rp, lp = oracle.token_index(np.array([0, B], np.int32), 1, B, False)
    assert rp.tolist() == [0] * B and lp.tolist() == list(range(B))


def test_token_index_rejects_bad_layouts():
    with pytest.raises(oracle.OracleError):
        oracle.token_index(np.array([0, 3, 2], np.int32), 2, 2, False)  # decreasing
    with pytest.raises(oracle.OracleError):
        oracle.token_index(np.array([0, 3], np.int32), 1, 4, False)  # cu[B] != T
    with pytest.raises(oracle.OracleError):
        oracle.token_index(None, 3, 4, True)  # decode needs B == T


# --------------------------------------------------------------------------
# brute force (no packed window, explicit interval walk) on many tiny batches


@pytest.mark.parametrize("chunk", range(8))
def test_oracle_matches_brute_force(chunk):
    for seed in range(chunk * 150, (chunk + 1) * 150):
        batch = wl.random_batch(seed, T_max=24)
        for reading in ("A", "B"):
            got = run_oracle(batch, reading)
            exp = run_brute(batch, reading)
            assert np.array_equal(got, exp), (seed, reading)


def test_reading_a_and_b_part_only_at_invalid_shifts():
    # with no boundary anywhere, every shift is valid and the readings agree
    for seed in range(40):
        batch = wl.random_batch(seed, density=0.0, boundary=10 ** 9)
        assert np.array_equal(run_oracle(batch, "A"), run_oracle(batch, "B"))


# --------------------------------------------------------------------------
# closed form for ngram_size 2


def test_ngram2_closed_form():
    """N=2, one head, no boundary, every token past its request's first:
    row = ((ids[t]*M0 XOR ids[t-1]*M1) mod v) + off, in uint64/int64 numpy."""
    rng = np.random.default_rng(5)
    for _ in range(50):
        T = int(rng.integers(2, 200))
        ids = rng.integers(0, wl.VOCAB, size=T, dtype=np.int64)
        ctx = rng.integers(0, wl.VOCAB, size=(1, 1), dtype=np.int64)
        M = wl.signed_multipliers(rng, 1, 2)
        v = int(wl.random_primes(rng, 1, 3, 2 ** 22)[0])
        off = int(rng.integers(0, 2 ** 40))
        batch = wl.Batch("n2", ids, ctx, np.array([0, T], np.int32), False, M,
                         np.array([[v]], np.int64), np.array([[off]], np.int64), 2, 1, -5)
        got = run_oracle(batch)[0, 1:, 0]
        u = ids.astype(np.uint64)
        with np.errstate(over="ignore"):
            mix = (u[1:] * np.uint64(int(M[0, 0]) % 2 ** 64)) ^ (u[:-1] * np.uint64(int(M[0, 1]) % 2 ** 64))
        exp = np.mod(mix.view(np.int64), v) + off
        assert np.array_equal(got, exp)


# --------------------------------------------------------------------------
# invariants of the definition


def test_rows_fall_in_their_head_range():
    # I1: off <= row < off + vocab for positive vocab and non-overflowing offsets
    for batch in [wl.prefill_512(), wl.decode(8), wl.ragged_16()]:
        out = run_oracle(batch)
        lo = batch.offsets[:, None, :]
        assert np.all(out >= lo) and np.all(out < lo + batch.vocab_sizes[:, None, :])


def test_vocab_one_gives_the_offset():
    # I2
    batch = wl.random_batch(3, T_max=40)
    batch.vocab_sizes[:] = 1
    assert np.array_equal(run_oracle(batch), np.broadcast_to(batch.offsets[:, None, :],
                                                            (batch.num_layers, batch.num_tokens,
                                                             batch.num_heads)))


def test_all_boundary_window_gives_one_row_per_head():
    # I3: every id the boundary -> every token hashes (b, b, ..., b)
    batch = wl.random_batch(9, T_max=40)
    batch.ids[:] = batch.boundary_id
    batch.ngram_context[:] = batch.boundary_id
    out = run_oracle(batch)
    assert np.all(out == out[:, :1, :])


@pytest.mark.parametrize("seed", range(12))
def test_chunked_prefill_equals_one_prefill(seed):
    # I4: the carried context makes the ids independent of chunking; this
    # also pins the context's column order (oldest id first)
    rng = np.random.default_rng(100 + seed)
    N = int(rng.integers(2, 7))
    full = wl.random_batch(1000 + seed, N=N, decode_batch=False, T_max=48)
    lengths = np.diff(full.cu_seqlens)
    r = int(np.argmax(lengths))
    T0 = int(lengths[r])
    assert T0 >= 2
    start = int(full.cu_seqlens[r])
    full = wl.Batch("f", full.ids[start:start + T0], full.ngram_context[r:r + 1],
                    np.array([0, T0], np.int32), False, full.layer_multipliers, full.vocab_sizes,
                    full.offsets, N, full.heads_per_ngram, full.boundary_id)
    k = int(rng.integers(1, T0))
    ids0 = full.ids[:T0]
    one = wl.Batch("one", ids0, full.ngram_context[:1], np.array([0, T0], np.int32), False,
                   full.layer_multipliers, full.vocab_sizes, full.offsets, N,
                   full.heads_per_ngram, full.boundary_id)
    a = wl.Batch("a", ids0[:k], full.ngram_context[:1], np.array([0, k], np.int32), False,
                 full.layer_multipliers, full.vocab_sizes, full.offsets, N, full.heads_per_ngram,
                 full.boundary_id)
    carried = np.concatenate([full.ngram_context[0], ids0[:k]])[-(N - 1):].reshape(1, N - 1)
    b = wl.Batch("b", ids0[k:], carried, np.array([0, T0 - k], np.int32), False,
                 full.layer_multipliers, full.vocab_sizes, full.offsets, N, full.heads_per_ngram,
                 full.boundary_id)
    assert np.array_equal(run_oracle(one), np.concatenate([run_oracle(a), run_oracle(b)], axis=1))


def test_decode_equals_one_token_prefills_and_differs_from_one_request():
    # I5
    batch = wl.decode(8)
    dec = run_oracle(batch)
    for t in range(8):
        single = wl.Batch("p", batch.ids[t:t + 1], batch.ngram_context[t:t + 1],
                          np.array([0, 1], np.int32), False, batch.layer_multipliers,
                          batch.vocab_sizes, batch.offsets, 3, 2, batch.boundary_id)
        assert np.array_equal(run_oracle(single)[:, 0], dec[:, t])
    one_req = wl.Batch("one", batch.ids, batch.ngram_context[:1], np.array([0, 8], np.int32), False,
                       batch.layer_multipliers, batch.vocab_sizes, batch.offsets, 3, 2,
                       batch.boundary_id)
    assert not np.array_equal(run_oracle(one_req), dec)
    # each decode context set to that token's sliding window -> equal
    ctx = np.concatenate([batch.ngram_context[0], batch.ids])
    slid = np.stack([ctx[t:t + 2] for t in range(8)])
    dec2 = wl.Batch("d2", batch.ids, slid, None, True, batch.layer_multipliers, batch.vocab_sizes,
                    batch.offsets, 3, 2, batch.boundary_id)
    assert np.array_equal(run_oracle(one_req), run_oracle(dec2))


def test_multilayer_slice_equals_single_layer():
    # I6
    batch = wl.random_batch(21, L=3, T_max=40)
    full = run_oracle(batch)
    for l in range(3):
        one = wl.Batch("l", batch.ids, batch.ngram_context, batch.cu_seqlens, batch.is_decode,
                       batch.layer_multipliers[l:l + 1], batch.vocab_sizes[l:l + 1],
                       batch.offsets[l:l + 1], batch.ngram_size, batch.heads_per_ngram,
                       batch.boundary_id)
        assert np.array_equal(run_oracle(one)[0], full[l])


def test_int32_ids_equal_int64_ids():
    # I7: int32 ids are sign-extended before hashing
    for seed in range(20):
        batch = wl.random_batch(seed)
        assert np.array_equal(run_oracle(batch), run_oracle(batch.with_ids_dtype(np.int32)))


# --------------------------------------------------------------------------
# the carried context


def test_next_context_is_the_tail_of_context_and_tokens():
    """Definition, written out with numpy: last N-1 of (context row, tokens)."""
    for seed in range(200):
        batch = wl.random_batch(seed, T_max=30)
        req, local = oracle.token_index(batch.cu_seqlens, batch.num_requests, batch.num_tokens,
                                        batch.is_decode)
        got = oracle.next_context(batch.ids, req, local, batch.ngram_context)
        C = batch.ngram_size - 1
        for r in range(batch.num_requests):
            toks = batch.ids[req == r]
            hist = np.concatenate([batch.ngram_context[r], toks])
            assert np.array_equal(got[r], hist[len(hist) - C:]), (seed, r)


@pytest.mark.parametrize("seed", range(8))
def test_carried_context_chains_chunks(seed):
    """I4 through the oracle's own carry: hashing a request in chunks, each
    chunk with the context the previous chunk carried, equals one prefill."""
    full = wl.random_batch(3000 + seed, decode_batch=False, T_max=60)
    lengths = np.diff(full.cu_seqlens)
    r = int(np.argmax(lengths))
    T0 = int(lengths[r])
    start = int(full.cu_seqlens[r])
    ids = full.ids[start:start + T0]
    one = wl.Batch("one", ids, full.ngram_context[r:r + 1], np.array([0, T0], np.int32), False,
                   full.layer_multipliers, full.vocab_sizes, full.offsets, full.ngram_size,
                   full.heads_per_ngram, full.boundary_id)
    rng = np.random.default_rng(seed)
    cuts = np.unique(np.concatenate([[0, T0], rng.integers(0, T0 + 1, size=3)]))
    ctx = full.ngram_context[r:r + 1]
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        chunk = wl.Batch("c", ids[a:b], ctx, np.array([0, b - a], np.int32), False,
                         full.layer_multipliers, full.vocab_sizes, full.offsets,
                         full.ngram_size, full.heads_per_ngram, full.boundary_id)
        parts.append(run_oracle(chunk))
        req, local = oracle.token_index(chunk.cu_seqlens, 1, chunk.num_tokens, False)
        ctx = oracle.next_context(chunk.ids, req, local, ctx)
    assert np.array_equal(np.concatenate(parts, axis=1), run_oracle(one))


# --------------------------------------------------------------------------
# the table gather (the row ids' consumer)


def oracle_embed(batch, table):
    req, local = oracle.token_index(batch.cu_seqlens, batch.num_requests, batch.num_tokens,
                                    batch.is_decode)
    return oracle.row_embed(batch.ids, req, local, batch.ngram_context, batch.layer_multipliers,
                            batch.vocab_sizes, batch.offsets, batch.ngram_size,
                            batch.heads_per_ngram, batch.boundary_id, table)


def test_embed_worked_example():
    g = json.load(open(GOLDEN))
    batch = golden_batch(g["setup"])
    V, D = g["embed"]["table_rows"], g["embed"]["dim"]
    vals = np.stack([np.arange(V), -2 * np.arange(V)], axis=1).astype(np.float32)
    table = wl.bf16_bits(vals).reshape(1, V, D)
    emb, _ = oracle_embed(batch, table)
    assert emb.tolist() == g["embed"]["expected"]


@pytest.mark.parametrize("seed", range(20))
def test_embed_of_a_row_valued_table_is_the_sum_of_row_ids(seed):
    """Row r of the table holds the value r (exact in bfloat16 below 256):
    the gathered sum is the sum of the (pinned) row ids over heads."""
    batch, _ = wl.small_table_batch(seed, D=3, T_max=40)
    rng = np.random.default_rng(seed)
    H = batch.num_heads
    batch.vocab_sizes[:] = rng.integers(1, max(2, 255 // H), size=batch.vocab_sizes.shape)
    batch.offsets[:] = wl.prefix_offsets(batch.vocab_sizes)
    V = int(batch.vocab_sizes.sum(axis=1).max())
    vals = np.repeat(np.arange(V, dtype=np.float32)[:, None], 3, axis=1)
    table = np.broadcast_to(wl.bf16_bits(vals), (batch.num_layers, V, 3)).copy()
    emb, _ = oracle_embed(batch, table)
    rows = run_oracle(batch)
    assert np.array_equal(emb[..., 0], rows.sum(axis=2).astype(np.float64))
    assert np.array_equal(emb[..., 1], emb[..., 0]) and np.array_equal(emb[..., 2], emb[..., 0])


@pytest.mark.parametrize("seed", range(10))
def test_embed_of_a_one_hot_table_counts_heads_per_row(seed):
    batch, _ = wl.small_table_batch(seed, T_max=30, L=2)
    batch.vocab_sizes[:] = np.minimum(batch.vocab_sizes, 17)
    batch.offsets[:] = wl.prefix_offsets(batch.vocab_sizes)
    V = int(batch.vocab_sizes.sum(axis=1).max())
    table = np.broadcast_to(wl.bf16_bits(np.eye(V, dtype=np.float32)),
                            (batch.num_layers, V, V)).copy()
    emb, _ = oracle_embed(batch, table)
    rows = run_oracle(batch)
    for l in range(batch.num_layers):
        for t in range(batch.num_tokens):
            counts = np.bincount(rows[l, t], minlength=V)[:V]
            assert np.array_equal(emb[l, t], counts.astype(np.float64))


@pytest.mark.parametrize("seed", range(10))
def test_embed_reads_each_layers_own_table(seed):
    """Layer l's table holds (l + 1) * r in row r (exact in bfloat16 up to
    256): each layer's gathered sum is (l + 1) times the sum of its row ids
    over heads, the row ids taken from the pure-Python brute force.  A gather
    that read another layer's table would scale the wrong sums."""
    batch, _ = wl.small_table_batch(seed, D=2, T_max=30, L=2)
    rng = np.random.default_rng(seed)
    H = batch.num_heads
    batch.vocab_sizes[:] = rng.integers(1, max(2, 127 // H), size=batch.vocab_sizes.shape)
    batch.offsets[:] = wl.prefix_offsets(batch.vocab_sizes)
    V = int(batch.vocab_sizes.sum(axis=1).max())
    L = batch.num_layers
    vals = (np.arange(L)[:, None] + 1) * np.arange(V)[None, :]
    table = wl.bf16_bits(np.repeat(vals[:, :, None], 2, axis=2).astype(np.float32))
    emb, _ = oracle_embed(batch, table)
    expect = (np.arange(L)[:, None] + 1) * run_brute(batch).sum(axis=2)
    assert np.array_equal(emb[..., 0], expect.astype(np.float64))
    assert np.array_equal(emb[..., 1], emb[..., 0])


@pytest.mark.parametrize("seed", range(5))
def test_embed_abs_sum_is_the_gather_of_magnitudes(seed):
    """The error-bound companion of the gather: the sum of |x| over the
    gathered values equals the gather of the table with its sign bits
    cleared."""
    batch, table = wl.small_table_batch(seed, D=8, T_max=30)
    _, abs_sum = oracle_embed(batch, table)
    magnitudes, _ = oracle_embed(batch, table & np.uint16(0x7FFF))
    assert np.array_equal(abs_sum, magnitudes)
    assert (table & np.uint16(0x8000)).any()  # the table has negative values to clear


def test_embed_rows_outside_the_table_add_nothing():
    batch, table = wl.small_table_batch(5, D=8, T_max=60)
    V = table.shape[1]
    cut = V // 2
    full, _ = oracle_embed(batch, np.concatenate(
        [table[:, :cut], np.zeros_like(table[:, cut:])], axis=1))
    short, _ = oracle_embed(batch, table[:, :cut])
    assert np.array_equal(full, short)


# --------------------------------------------------------------------------
# geometry preconditions ("Why it is safe", last point) and domain errors


def test_oracle_refuses_bad_geometry_and_zero_vocab():
    batch = wl.prefill_512()
    req, local = oracle.token_index(batch.cu_seqlens, 1, batch.num_tokens, False)
    args = dict(input_ids=batch.ids, req=req, local=local, layer_multipliers=batch.layer_multipliers,
                offsets=batch.offsets, ngram_size=3, heads_per_ngram=2, boundary_id=batch.boundary_id)
    with pytest.raises(oracle.OracleError) as e:
        oracle.row_ids(ngram_context=np.zeros((1, 3), np.int64), vocab_sizes=batch.vocab_sizes, **args)
    assert e.value.code == oracle.ORC_ERR_GEOMETRY
    with pytest.raises(oracle.OracleError) as e:
        oracle.row_ids(ngram_context=batch.ngram_context, vocab_sizes=batch.vocab_sizes,
                       **{**args, "heads_per_ngram": 1})
    assert e.value.code == oracle.ORC_ERR_GEOMETRY
    v = batch.vocab_sizes.copy()
    v[0, 1] = 0
    with pytest.raises(oracle.OracleError) as e:
        oracle.row_ids(ngram_context=batch.ngram_context, vocab_sizes=v, **args)
    assert e.value.code == oracle.ORC_ERR_VOCAB
    bad_local = local.copy()
    bad_local[5] = 7
    with pytest.raises(oracle.OracleError) as e:
        oracle.row_ids(ngram_context=batch.ngram_context, vocab_sizes=batch.vocab_sizes,
                       **{**args, "local": bad_local})
    assert e.value.code == oracle.ORC_ERR_INDEX
