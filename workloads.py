"""Seeded synthetic inputs for the PLE n-gram row-id hash.

This module only draws inputs (ids, batch layouts, contexts, multipliers,
vocab sizes, offsets).  It holds none of the hash arithmetic and imports
neither the CUDA binding nor the oracle, so both sides can be fed from it.

The workloads follow the shapes and value distributions of the PLE layer
described in FreeToken PR #338 ("perf(ple): fuse the n-gram row-id hash into
one Triton kernel", sections "What" and "Measured"): token ids from a
151936-entry vocabulary, boundary id 151643, ngram_size - 1 ids of carried
context per request, per-layer signed int64 multipliers, prime head vocab
sizes and prefix-sum head offsets.  There is no public dataset for this path;
every array is synthetic and seeded (seed = config index * 1000 + replay).
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

VOCAB = 151936
BOUNDARY = 151643
I64_MIN = -(2 ** 63)
I64_MAX = 2 ** 63 - 1


@dataclass
class Batch:
    name: str
    ids: np.ndarray            # [T] int32 or int64
    ngram_context: np.ndarray  # [B, N-1], same dtype as ids
    cu_seqlens: np.ndarray | None  # [B+1] int32, None for a decode
    is_decode: bool
    layer_multipliers: np.ndarray  # [L, N] int64
    vocab_sizes: np.ndarray        # [L, H] int64
    offsets: np.ndarray            # [L, H] int64
    ngram_size: int
    heads_per_ngram: int
    boundary_id: int = BOUNDARY
    meta: dict = field(default_factory=dict)

    @property
    def num_tokens(self) -> int:
        return int(self.ids.shape[0])

    @property
    def num_requests(self) -> int:
        return int(self.ngram_context.shape[0])

    @property
    def num_layers(self) -> int:
        return int(self.layer_multipliers.shape[0])

    @property
    def num_heads(self) -> int:
        return int(self.vocab_sizes.shape[1])

    @property
    def row_ids_per_call(self) -> int:
        return self.num_layers * self.num_tokens * self.num_heads

    def algorithmic_bytes(self) -> int:
        """Bytes the method must move for one call: ids, the (req, local)
        index and the context read, row ids written, parameters read."""
        idb = self.ids.dtype.itemsize
        T, B, L, H, N = (self.num_tokens, self.num_requests, self.num_layers, self.num_heads,
                         self.ngram_size)
        return T * (idb + 8 + 8 * L * H) + B * (N - 1) * idb + 8 * L * (N + 2 * H)

    def with_ids_dtype(self, dtype) -> "Batch":
        return replace(self, ids=self.ids.astype(dtype),
                       ngram_context=self.ngram_context.astype(dtype))


# ----------------------------------------------------------------------------
# primitive draws


def _small_primes(limit: int) -> np.ndarray:
    sieve = np.ones(limit + 1, dtype=bool)
    sieve[:2] = False
    for i in range(2, int(limit ** 0.5) + 1):
        if sieve[i]:
            sieve[i * i::i] = False
    return np.nonzero(sieve)[0].astype(np.int64)


def random_primes(rng: np.random.Generator, n: int, lo: int, hi: int) -> np.ndarray:
    """n primes drawn uniformly from the primes in [lo, hi) (hi <= 2**40)."""
    ps = _small_primes(int(hi ** 0.5) + 1)
    out = []
    while len(out) < n:
        cand = rng.integers(lo, hi, size=max(64, 8 * n), dtype=np.int64)
        ok = np.ones(cand.shape, dtype=bool)
        for p in ps:
            ok &= (cand % p != 0) | (cand == p)
        out.extend(int(c) for c in cand[ok & (cand >= 2)])
    return np.array(out[:n], dtype=np.int64)


def signed_multipliers(rng: np.random.Generator, L: int, N: int) -> np.ndarray:
    """Uniform over the whole signed int64 range (random 64 bits)."""
    return rng.integers(I64_MIN, I64_MAX, size=(L, N), dtype=np.int64, endpoint=True)


def prefix_offsets(vocab: np.ndarray) -> np.ndarray:
    """Exclusive prefix sum of the head vocab sizes, per layer."""
    off = np.zeros_like(vocab)
    off[:, 1:] = np.cumsum(vocab[:, :-1], axis=1)
    return off


def uniform_ids(rng, n, density=0.0, boundary=BOUNDARY):
    ids = rng.integers(0, VOCAB, size=n, dtype=np.int64)
    if density > 0:
        ids[rng.random(n) < density] = boundary
    return ids


def random_split(rng: np.random.Generator, total: int, parts: int) -> np.ndarray:
    """A uniformly drawn composition of `total` into `parts` positive parts."""
    cuts = np.sort(rng.choice(np.arange(1, total), size=parts - 1, replace=False))
    edges = np.concatenate([[0], cuts, [total]])
    return np.diff(edges).astype(np.int64)


def cu_from_lengths(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu


def boundary_runs(rng, ids, density, max_run, boundary=BOUNDARY):
    """Overwrite runs of length U[1, max_run] with the boundary id, at uniform
    start positions, until `density` of the ids are boundaries."""
    n = ids.shape[0]
    target = int(np.ceil(density * n))
    count = int((ids == boundary).sum())
    while count < target:
        k = max(16, (target - count) // max_run + 1)
        starts = rng.integers(0, n, size=k)
        lens = rng.integers(1, max_run + 1, size=k)
        for s, ln in zip(starts, lens):
            ids[s:s + ln] = boundary
        count = int((ids == boundary).sum())
    return ids


def _params(rng, L, N, hpn, lo, hi):
    H = (N - 1) * hpn
    vocab = random_primes(rng, L * H, lo, hi).reshape(L, H)
    return signed_multipliers(rng, L, N), vocab, prefix_offsets(vocab)


# ----------------------------------------------------------------------------
# the five workloads of the PLE row-id hash


def prefill_512(replay: int = 0) -> Batch:
    """One request, T=512 int64 ids U[0,151936) with 1% boundaries,
    ngram_size 3, 2 heads per order (4 heads), one layer, [1, 2] context."""
    rng = np.random.default_rng(0 * 1000 + replay)
    N, hpn, L, T = 3, 2, 1, 512
    M, vocab, off = _params(rng, L, N, hpn, 2 ** 17, 2 ** 20)
    ids = uniform_ids(rng, T, 0.01)
    ctx = uniform_ids(rng, N - 1).reshape(1, N - 1)
    return Batch("prefill_512", ids, ctx, cu_from_lengths([T]), False, M, vocab, off, N, hpn)


def decode(B: int, replay: int = 0) -> Batch:
    """B requests, one token each at offset 0; [B, 2] context with 5%
    boundaries; ngram_size 3, 4 heads, one layer.  The parameters stay fixed
    across replays; ids and context are fresh per replay."""
    prng = np.random.default_rng(1 * 1000)
    N, hpn, L = 3, 2, 1
    M, vocab, off = _params(prng, L, N, hpn, 2 ** 17, 2 ** 20)
    rng = np.random.default_rng(1 * 1000 + 1 + replay * 16 + B)
    ids = uniform_ids(rng, B)
    ctx = uniform_ids(rng, B * (N - 1), 0.05).reshape(B, N - 1)
    return Batch(f"decode_b{B}", ids, ctx, None, True, M, vocab, off, N, hpn, meta={"replay": replay})


def ragged_16(replay: int = 0) -> Batch:
    """16 requests with lengths U[1,4096] (int32 cu_seqlens), 2% boundaries,
    ngram_size 3, 4 heads per order (8 heads), one layer."""
    rng = np.random.default_rng(2 * 1000 + replay)
    N, hpn, L, B = 3, 4, 1, 16
    M, vocab, off = _params(rng, L, N, hpn, 2 ** 17, 2 ** 20)
    lengths = rng.integers(1, 4097, size=B)
    T = int(lengths.sum())
    ids = uniform_ids(rng, T, 0.02)
    ctx = uniform_ids(rng, B * (N - 1), 0.02).reshape(B, N - 1)
    return Batch("ragged_16", ids, ctx, cu_from_lengths(lengths), False, M, vocab, off, N, hpn)


def mixed_8192(replay: int = 0) -> Batch:
    """T=8192: 8 prefills (a random split of 7936) and 256 one-token decodes
    in one cu_seqlens, requests in random order; 2% boundaries (the workload
    names no density); ngram_size 5, 8 heads per order (32 heads), 48 layers
    emitted in one call; vocab primes in [2^16, 2^22)."""
    rng = np.random.default_rng(3 * 1000 + replay)
    N, hpn, L = 5, 8, 48
    M, vocab, off = _params(rng, L, N, hpn, 2 ** 16, 2 ** 22)
    lengths = np.concatenate([random_split(rng, 7936, 8), np.ones(256, dtype=np.int64)])
    lengths = lengths[rng.permutation(lengths.shape[0])]
    B = lengths.shape[0]
    T = int(lengths.sum())
    ids = uniform_ids(rng, T, 0.02)
    ctx = uniform_ids(rng, B * (N - 1), 0.02).reshape(B, N - 1)
    return Batch("mixed_8192", ids, ctx, cu_from_lengths(lengths), False, M, vocab, off, N, hpn)


def prefill_262144(replay: int = 0, ids_dtype=np.int64, context_all_boundary: bool = False) -> Batch:
    """T=262144 in 4 requests (a random split); ngram_size 4, 4 heads per
    order (12 heads), 8 layers; adversarial boundaries: runs of length
    U[1,8] until 20% of the ids are the boundary id, plus a boundary at every
    request start; context rows U with 20% boundaries (or, in the second
    reading of "boundary at every request start", all boundaries)."""
    rng = np.random.default_rng(4 * 1000 + replay)
    N, hpn, L, B, T = 4, 4, 8, 4, 262144
    M, vocab, off = _params(rng, L, N, hpn, 2 ** 17, 2 ** 20)
    lengths = random_split(rng, T, B)
    cu = cu_from_lengths(lengths)
    ids = boundary_runs(rng, uniform_ids(rng, T), 0.20, 8)
    ids[cu[:-1]] = BOUNDARY
    if context_all_boundary:
        ctx = np.full((B, N - 1), BOUNDARY, dtype=np.int64)
    else:
        ctx = uniform_ids(rng, B * (N - 1), 0.20).reshape(B, N - 1)
    name = "prefill_262144" + ("_ctxb" if context_all_boundary else "")
    batch = Batch(name, ids, ctx, cu, False, M, vocab, off, N, hpn)
    return batch.with_ids_dtype(ids_dtype) if ids_dtype != np.int64 else batch


def prefill_262144_lowrep(replay: int = 0) -> Batch:
    """The large prefill's shape (T=262144 in 4 requests, ngram_size 4,
    12 heads, 8 layers) with the ragged and mixed batches' boundary density:
    2% isolated boundary ids at uniform positions (no runs), so that windows,
    and the row ids they hash to, rarely repeat -- the input for measuring
    the table gather's random-row rate without repeated rows served from L2."""
    rng = np.random.default_rng(5 * 1000 + replay)
    N, hpn, L, B, T = 4, 4, 8, 4, 262144
    M, vocab, off = _params(rng, L, N, hpn, 2 ** 17, 2 ** 20)
    cu = cu_from_lengths(random_split(rng, T, B))
    ids = uniform_ids(rng, T, 0.02)
    ctx = uniform_ids(rng, B * (N - 1), 0.02).reshape(B, N - 1)
    return Batch("prefill_262144_lowrep", ids, ctx, cu, False, M, vocab, off, N, hpn)


def all_workloads(replay: int = 0):
    """Every configuration the hash is checked on, small first."""
    out = [prefill_512(replay)]
    out += [decode(B, replay) for B in (1, 4, 8)]
    out += [ragged_16(replay), mixed_8192(replay), prefill_262144(replay),
            prefill_262144(replay, np.int32), prefill_262144(replay, context_all_boundary=True)]
    return out


# ----------------------------------------------------------------------------
# small random batches for edge-case and property checks

EDGE_VOCABS = [1, 2, 3, 7, 11, 2 ** 31 - 1, 2 ** 31, 2 ** 31 + 1, 2 ** 32 - 1, 2 ** 32, 2 ** 32 + 15,
               2 ** 40 + 7, 2 ** 62 + 3, I64_MAX, -1, -2, -7, -(2 ** 31), -(2 ** 40) - 1, I64_MIN]


def random_batch(seed: int, T_max: int = 64, N=None, hpn=None, L=None, density=None,
                 ids_dtype=np.int64, decode_batch=None, vocab_mode: str = "mixed",
                 boundary=None) -> Batch:
    """A small random ragged batch (empty requests allowed) with adversarial
    parameters: full-range signed multipliers (INT64_MIN/MAX included), vocab
    sizes mixing primes, tiny values, values at the 2^31 / 2^32 edges and
    negative values (torch.remainder's floored rule), boundary densities from
    0 to 1.  ids are small so that collisions with the boundary id are common
    when the boundary is drawn from the same range."""
    rng = np.random.default_rng(seed)
    N = int(rng.integers(2, 9)) if N is None else N
    hpn = int(rng.integers(1, 4)) if hpn is None else hpn
    L = int(rng.integers(1, 4)) if L is None else L
    H = (N - 1) * hpn
    if density is None:
        density = float(rng.choice([0.0, 0.1, 0.3, 0.5, 1.0]))
    is_decode = bool(rng.random() < 0.2) if decode_batch is None else decode_batch
    if is_decode:
        T = int(rng.integers(1, T_max + 1))
        B = T
        cu = None
    else:
        B = int(rng.integers(1, 9))
        lengths = rng.integers(0, max(2, 2 * T_max // B), size=B)
        if lengths.sum() == 0:
            lengths[rng.integers(0, B)] = 1
        T = int(lengths.sum())
        cu = cu_from_lengths(lengths)
    lo_id, hi_id = (-50, 50) if rng.random() < 0.5 else (0, VOCAB)
    b = int(rng.integers(lo_id, hi_id)) if boundary is None else boundary
    ids = rng.integers(lo_id, hi_id, size=T, dtype=np.int64)
    ids[rng.random(T) < density] = b
    ctx = rng.integers(lo_id, hi_id, size=(B, N - 1), dtype=np.int64)
    ctx[rng.random((B, N - 1)) < density] = b
    M = signed_multipliers(rng, L, N)
    M[rng.random((L, N)) < 0.1] = I64_MIN
    M[rng.random((L, N)) < 0.1] = I64_MAX
    if vocab_mode == "primes":
        vocab = random_primes(rng, L * H, 2 ** 16, 2 ** 22).reshape(L, H)
    else:
        pick = rng.random((L, H))
        vocab = random_primes(rng, L * H, 2, 2 ** 22).reshape(L, H)
        edge = rng.choice(np.array(EDGE_VOCABS, dtype=np.int64), size=(L, H))
        vocab = np.where(pick < 0.5, edge, vocab)
    off = rng.integers(I64_MIN, I64_MAX, size=(L, H), dtype=np.int64, endpoint=True)
    off = np.where(rng.random((L, H)) < 0.5, prefix_offsets(np.abs(vocab) % 2 ** 40), off)
    batch = Batch(f"random_{seed}", ids, ctx, cu, is_decode, M, vocab, off, N, hpn, b,
                  meta={"density": density})
    return batch.with_ids_dtype(ids_dtype) if ids_dtype != np.int64 else batch


def slice_batch(batch: Batch, start: int, stop: int) -> Batch:
    """The tokens [start, stop) of a prefill batch as a batch of their own.

    A request cut at `start` continues with a carried context: the last N-1
    ids of (its context followed by its tokens before `start`), which is the
    state the page's ngram_context carries from one call to the next, so the
    slice's row ids equal the corresponding rows of the whole batch.  Only
    ids are moved here; nothing is hashed.
    """
    if batch.is_decode:
        ids = batch.ids[start:stop]
        return replace(batch, name=f"{batch.name}[{start}:{stop}]", ids=ids,
                       ngram_context=batch.ngram_context[start:stop])
    C = batch.ngram_size - 1
    cu = batch.cu_seqlens.astype(np.int64)
    r_first = int(np.searchsorted(cu, start, side="right") - 1)
    r_last = int(np.searchsorted(cu, max(stop - 1, start), side="right") - 1)
    lengths, ctx_rows = [], []
    for r in range(r_first, r_last + 1):
        a, b = max(int(cu[r]), start), min(int(cu[r + 1]), stop)
        if a > b:
            a = b
        lengths.append(b - a)
        hist = np.concatenate([batch.ngram_context[r], batch.ids[int(cu[r]):a]])
        ctx_rows.append(hist[len(hist) - C:])
    ctx = np.stack(ctx_rows).astype(batch.ngram_context.dtype)
    return replace(batch, name=f"{batch.name}[{start}:{stop}]", ids=batch.ids[start:stop],
                   ngram_context=ctx, cu_seqlens=cu_from_lengths(lengths))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 values to bfloat16 bit patterns (uint16), rounding to nearest
    even.  Input construction only."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def embed_table(rng: np.random.Generator, L: int, V: int, D: int) -> np.ndarray:
    """A synthetic per-layer embedding table [L, V, D] of bfloat16 bits with
    standard-normal values (no trained weights exist for this path)."""
    return bf16_bits(rng.standard_normal((L, V, D), dtype=np.float32))


def small_table_batch(seed: int, D: int = 16, T_max: int = 100, N=None, hpn=None, L=None,
                      ids_dtype=np.int64, decode_batch=None) -> tuple:
    """A random batch whose heads index a small table (vocab primes below
    2^12, prefix-sum offsets), with that table; V is the largest per-layer
    vocab total, so every row id is in range unless the caller shrinks V."""
    batch = random_batch(seed, T_max=T_max, N=N, hpn=hpn, L=L, ids_dtype=ids_dtype,
                         decode_batch=decode_batch)
    rng = np.random.default_rng(seed + 1)
    H = batch.num_heads
    vocab = random_primes(rng, batch.num_layers * H, 2, 2 ** 12).reshape(batch.num_layers, H)
    batch = replace(batch, vocab_sizes=vocab, offsets=prefix_offsets(vocab))
    V = int(vocab.sum(axis=1).max())
    return batch, embed_table(rng, batch.num_layers, V, D)
