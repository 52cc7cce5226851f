"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a private copy of oracle/ple_oracle.c (a
dropped term, a wrong sign, an index off by one, a transposed operand, a
reversed order), compiles it with gcc into a temporary directory, and runs
the pin battery against it: the hand-worked window under both readings, the
sign/wrap cases, and the pure-Python brute force on random batches.  A
mutant that passes every pin would mean the pins leave that part of the
oracle unchecked, so each one must fail at least one pin.

The oracle's other functions -- the token index, the carried context and
the table gather -- have planted mistakes of their own, each run against the
pins of that function (written out here against definitions that do not
call the function under test: numpy's searchsorted for the index, the tail
of context and tokens for the carry, the brute-force row ids for the
gather).

The eos fill of the packed window is not mutated: with ctx_len = N-1 no
token reads a cell left of its request's context, and cells right of a
request's last token are never read, so the fill value cannot change a row
id (an equivalent mutant, not a mistake).
"""

import ctypes
import json
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import workloads as wl
from brute_force import brute_row_ids

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ple_oracle.c")
GOLDEN = os.path.join(ROOT, "tests", "golden", "worked_example.json")

MUTANTS = {
    "xor_becomes_or": ("mix ^= wrap_mul(", "mix |= wrap_mul("),
    "order_drops_last_shift": ("for (int32_t s = 0; s < n; ++s) mix",
                               "for (int32_t s = 0; s < n - 1; ++s) mix"),
    "multipliers_reversed": ("wrap_mul(V[s], M[(int64_t)l * N + s])",
                             "wrap_mul(V[s], M[(int64_t)l * N + (N - 1 - s)])"),
    "truncated_remainder": ("if (r != 0 && ((r < 0) != (v < 0))) r += v;", ""),
    "validity_ignored": ("V[s] = invalid_as_zero ? 0 : b;", "V[s] = row[p - s];"),
    "token_itself_checked": ("lastb[r * width + p - 1] < p - s", "lastb[r * width + p] < p - s"),
    "interval_one_short": ("lastb[r * width + p - 1] < p - s", "lastb[r * width + p - 1] <= p - s"),
    "context_reversed": ("load_id(ngram_context, id_bytes, (int64_t)r * ctx_len + c)",
                         "load_id(ngram_context, id_bytes, (int64_t)r * ctx_len + (ctx_len - 1 - c))"),
    "offset_dropped": ("wrap_add(oracle_floor_mod(mix, vocab[k]), off[k])",
                       "oracle_floor_mod(mix, vocab[k])"),
    "offset_subtracted": ("wrap_add(oracle_floor_mod(mix, vocab[k]), off[k])",
                          "wrap_add(oracle_floor_mod(mix, vocab[k]), -off[k])"),
    "heads_head_major": ("const int64_t h = (int64_t)(n - 2) * hpn + j;",
                         "const int64_t h = (int64_t)j * (N - 1) + (n - 2);"),
    "int32_zero_extended": ("return (int64_t)((const int32_t*)p)[i];",
                            "return (int64_t)(uint32_t)((const int32_t*)p)[i];"),
    "out_token_major": ("out[((int64_t)l * T + t) * H + h]", "out[((int64_t)t * L + l) * H + h]"),
    "mix_seeded_with_one": ("int64_t mix = 0;", "int64_t mix = 1;"),
    "sign_fix_wrong_way": ("if (r != 0 && ((r < 0) != (v < 0))) r += v;",
                           "if (r != 0 && ((r < 0) != (v < 0))) r -= v;"),
}


class Mutant:
    def __init__(self, path):
        self.lib = ctypes.CDLL(path)
        p, i32, i64, c = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int
        self.lib.oracle_token_index.argtypes = [p, i32, i64, c, p, p]
        args = [p, c, i64, p, p, p, i32, i32, p, p, p, i32, i32, i32, i32, i64, p]
        for n in ("oracle_row_ids", "oracle_row_ids_reading_b"):
            getattr(self.lib, n).argtypes = args

    def rows(self, batch, reading="A"):
        T = batch.num_tokens
        req = np.zeros(T, np.int32)
        local = np.zeros(T, np.int32)
        cu = batch.cu_seqlens
        self.lib.oracle_token_index(cu.ctypes.data if cu is not None else None,
                                    batch.num_requests, T, int(batch.is_decode),
                                    req.ctypes.data, local.ctypes.data)
        ids = np.ascontiguousarray(batch.ids)
        ctx = np.ascontiguousarray(batch.ngram_context, dtype=ids.dtype)
        M = np.ascontiguousarray(batch.layer_multipliers)
        vocab = np.ascontiguousarray(batch.vocab_sizes)
        off = np.ascontiguousarray(batch.offsets)
        out = np.zeros((batch.num_layers, T, batch.num_heads), np.int64)
        fn = self.lib.oracle_row_ids if reading == "A" else self.lib.oracle_row_ids_reading_b
        rc = fn(ids.ctypes.data, ids.dtype.itemsize, T, req.ctypes.data, local.ctypes.data,
                ctx.ctypes.data, batch.num_requests, batch.ngram_size - 1, M.ctypes.data,
                vocab.ctypes.data, off.ctypes.data, batch.num_heads, batch.ngram_size,
                batch.heads_per_ngram, batch.num_layers, batch.boundary_id, out.ctypes.data)
        return out if rc == 0 else None


def golden(d):
    return wl.Batch("g", np.array(d["input_ids"], np.int64), np.array(d["ngram_context"], np.int64),
                    np.array(d["cu_seqlens"], np.int32), False,
                    np.array(d["layer_multipliers"], np.int64), np.array(d["vocab_sizes"], np.int64),
                    np.array(d["offsets"], np.int64), d["ngram_size"], d["heads_per_ngram"],
                    d["boundary_id"])


def pins_fail(m: Mutant) -> str | None:
    """Name of the first pin the oracle under test fails, or None."""
    g = json.load(open(GOLDEN))
    b = golden(g["setup"])
    out = m.rows(b, "A")
    if out is None or out.tolist() != g["expected_reading_a"]:
        return "worked example (A)"
    out = m.rows(b, "B")
    if out is None or out.tolist() != g["expected_reading_b"]:
        return "worked example (B)"
    for d in g["sign_and_wrap"]:
        out = m.rows(golden(d))
        if out is None or out.tolist() != d["expected"]:
            return "sign/wrap"
    for seed in range(120):
        dtype = np.int32 if seed % 4 == 0 else np.int64
        batch = wl.random_batch(seed, T_max=20, ids_dtype=dtype)
        from oracle import token_index  # the index is pinned separately
        req, local = token_index(batch.cu_seqlens, batch.num_requests, batch.num_tokens,
                                 batch.is_decode)
        exp = np.array(brute_row_ids(batch.ids, req, local, batch.ngram_context,
                                     batch.layer_multipliers, batch.vocab_sizes, batch.offsets,
                                     batch.ngram_size, batch.heads_per_ngram, batch.boundary_id),
                       dtype=np.int64)
        out = m.rows(batch)
        if out is None or not np.array_equal(out, exp):
            return f"brute force (seed {seed})"
    return None


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory() as d:
        yield d


def build_variant(workdir, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    path_c = os.path.join(workdir, f"{name}.c")
    path_so = os.path.join(workdir, f"{name}.so")
    with open(path_c, "w") as fh:
        fh.write(src.replace(old, new))
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-w", "-o", path_so, path_c],
                   check=True)
    return Mutant(path_so)


def test_unmutated_copy_passes_every_pin(workdir):
    assert pins_fail(build_variant(workdir, "clean", "#include <stdint.h>",
                                   "#include <stdint.h>")) is None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(workdir, name):
    old, new = MUTANTS[name]
    assert pins_fail(build_variant(workdir, name, old, new)) is not None, \
        f"no pin catches the mutant {name}"


# --------------------------------------------------------------------------
# the token index, the carried context and the table gather


def mutate(src: str, anchor: str, old: str, new: str) -> str:
    """src with the first `old` after `anchor` replaced by `new`."""
    i = src.index(old, src.index(anchor))
    return src[:i] + new + src[i + len(old):]


INDEX = "int oracle_token_index("
CARRY = "int oracle_next_context("
EMBED = "int oracle_row_embed("
BF16 = "static double bf16_to_double("

FUNCTION_MUTANTS = {
    "index_offset_not_rebased": ("index", INDEX, "local[t] = t - cu_seqlens[r];", "local[t] = t;"),
    "index_request_shifted": ("index", INDEX, "req[t] = r;", "req[t] = r + 1;"),
    "index_last_request_dropped": ("index", INDEX, "for (int32_t r = 0; r < num_requests; ++r) {",
                                   "for (int32_t r = 0; r < num_requests - 1; ++r) {"),
    "index_decode_offset_one": ("index", INDEX, "local[t] = 0;", "local[t] = 1;"),
    "index_decode_one_request": ("index", INDEX, "req[t] = (int32_t)t;", "req[t] = 0;"),
    "index_order_unchecked": ("index", INDEX,
                              "if (cu_seqlens[r + 1] < cu_seqlens[r]) return ORC_ERR_INDEX;", ""),
    "carry_newest_first": ("carry", CARRY, "const int64_t v = seq[n - ctx_len + c];",
                           "const int64_t v = seq[n - 1 - c];"),
    "carry_keeps_old_row": ("carry", CARRY, "const int64_t v = seq[n - ctx_len + c];",
                            "const int64_t v = seq[c];"),
    "carry_tokens_from_batch_start": ("carry", CARRY, "load_id(input_ids, id_bytes, start[r] + i)",
                                      "load_id(input_ids, id_bytes, i)"),
    "carry_context_reversed": ("carry", CARRY, "(int64_t)r * ctx_len + c);",
                               "(int64_t)r * ctx_len + (ctx_len - 1 - c));"),
    "embed_skips_last_head": ("embed", EMBED, "for (int32_t h = 0; h < H; ++h) {",
                              "for (int32_t h = 0; h < H - 1; ++h) {"),
    "embed_first_layer_table": ("embed", EMBED, "table + ((int64_t)l * V + row) * D",
                                "table + ((int64_t)0 * V + row) * D"),
    "embed_drops_last_row": ("embed", EMBED, "if (row < 0 || row >= V) continue;",
                             "if (row < 0 || row >= V - 1) continue;"),
    "embed_abs_keeps_sign": ("embed", EMBED, "a[d] += x < 0 ? -x : x;", "a[d] += x;"),
    "embed_token_major_out": ("embed", EMBED, "double* o = out + ((int64_t)l * T + t) * D;",
                              "double* o = out + ((int64_t)t * L + l) * D;"),
    "embed_bf16_shift": ("embed", BF16, "(uint32_t)bits << 16", "(uint32_t)bits << 15"),
}


def build_function_variant(workdir, name, anchor, old, new):
    path_c = os.path.join(workdir, f"{name}.c")
    path_so = os.path.join(workdir, f"{name}.so")
    with open(path_c, "w") as fh:
        fh.write(mutate(open(SRC).read(), anchor, old, new))
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-w", "-o", path_so, path_c],
                   check=True)
    return path_so


def searchsorted_index(cu, B, T, is_decode):
    """(req, local) from the definition: the last r with cu[r] <= t."""
    t = np.arange(T)
    if is_decode:
        return t.astype(np.int32), np.zeros(T, np.int32)
    owner = np.searchsorted(np.asarray(cu), t, side="right") - 1
    return owner.astype(np.int32), (t - np.asarray(cu)[owner]).astype(np.int32)


def index_pins_fail(path) -> str | None:
    """The index against numpy's searchsorted, the decode rule, and refused
    layouts; every call gets 64 spare entries past T (a planted mistake may
    write there, and that is caught, never a write out of bounds)."""
    lib = oracle.load_library(path)

    def call(cu, B, T, decode):
        req = np.full(T + 64, -7, np.int32)
        local = np.full(T + 64, -7, np.int32)
        rc = lib.oracle_token_index(cu.ctypes.data if cu is not None else None, B, T,
                                    int(decode), req.ctypes.data, local.ctypes.data)
        return rc, req, local

    rng = np.random.default_rng(11)
    for _ in range(80):
        B = int(rng.integers(1, 9))
        cu = np.concatenate([[0], np.cumsum(rng.integers(0, 6, size=B))]).astype(np.int32)
        T = int(cu[-1])
        if T == 0:
            continue
        rc, req, local = call(cu, B, T, False)
        er, el = searchsorted_index(cu, B, T, False)
        if (rc != 0 or not np.array_equal(req[:T], er) or not np.array_equal(local[:T], el)
                or (req[T:] != -7).any() or (local[T:] != -7).any()):
            return "prefill index against searchsorted"
    for B in (1, 3, 8):
        rc, req, local = call(None, B, B, True)
        if rc != 0 or not np.array_equal(req[:B], np.arange(B)) or local[:B].any():
            return "decode index"
    for cu, B, T in ((np.array([0, 3, 2], np.int32), 2, 2), (np.array([0, 3], np.int32), 1, 4),
                     (np.array([0, 2, 1, 3], np.int32), 3, 3)):
        if call(cu, B, T, False)[0] == 0:
            return "malformed layout accepted"
    return None


def carry_pins_fail(path) -> str | None:
    """The carried context against the tail of (context row, tokens)."""
    with oracle.using_library(path):
        for seed in range(80):
            b = wl.random_batch(seed, T_max=30)
            req, local = searchsorted_index(b.cu_seqlens, b.num_requests, b.num_tokens,
                                            b.is_decode)
            got = oracle.next_context(b.ids, req, local, b.ngram_context)
            C = b.ngram_size - 1
            for r in range(b.num_requests):
                hist = np.concatenate([b.ngram_context[r], b.ids[req == r]])
                if not np.array_equal(got[r], hist[len(hist) - C:]):
                    return f"tail of context and tokens (seed {seed})"
    return None


def embed_pins_fail(path) -> str | None:
    """The gather against the hand-worked example and against sums of the
    brute-force row ids: row-valued tables distinct per layer, one-hot
    tables, and the sum of magnitudes."""
    g = json.load(open(GOLDEN))
    with oracle.using_library(path):
        def gather(b, table):
            req, local = searchsorted_index(b.cu_seqlens, b.num_requests, b.num_tokens,
                                            b.is_decode)
            return oracle.row_embed(b.ids, req, local, b.ngram_context, b.layer_multipliers,
                                    b.vocab_sizes, b.offsets, b.ngram_size, b.heads_per_ngram,
                                    b.boundary_id, table)

        def rows(b):
            req, local = searchsorted_index(b.cu_seqlens, b.num_requests, b.num_tokens,
                                            b.is_decode)
            return np.array(brute_row_ids(b.ids, req, local, b.ngram_context,
                                          b.layer_multipliers, b.vocab_sizes, b.offsets,
                                          b.ngram_size, b.heads_per_ngram, b.boundary_id),
                            dtype=np.int64).reshape(b.num_layers, b.num_tokens, b.num_heads)

        b = golden(g["setup"])
        V, D = g["embed"]["table_rows"], g["embed"]["dim"]
        vals = np.stack([np.arange(V), -2 * np.arange(V)], axis=1).astype(np.float32)
        if gather(b, wl.bf16_bits(vals).reshape(1, V, D))[0].tolist() != g["embed"]["expected"]:
            return "worked example"
        for seed in range(8):
            b, table = wl.small_table_batch(seed, D=2, T_max=24, L=2)
            rng = np.random.default_rng(seed)
            H = b.num_heads
            b.vocab_sizes[:] = rng.integers(1, max(2, 127 // H), size=b.vocab_sizes.shape)
            b.offsets[:] = wl.prefix_offsets(b.vocab_sizes)
            V = int(b.vocab_sizes.sum(axis=1).max())
            L = b.num_layers
            scaled = (np.arange(L)[:, None] + 1) * np.arange(V)[None, :]
            tab = wl.bf16_bits(np.repeat(scaled[:, :, None], 2, axis=2).astype(np.float32))
            r = rows(b)
            emb, _ = gather(b, tab)
            if not np.array_equal(emb[..., 0], ((np.arange(L)[:, None] + 1) * r.sum(axis=2))):
                return f"row-valued tables (seed {seed})"
            eye = np.broadcast_to(wl.bf16_bits(np.eye(V, dtype=np.float32)), (L, V, V)).copy()
            emb, _ = gather(b, eye)
            for l in range(L):
                for t in range(b.num_tokens):
                    if not np.array_equal(emb[l, t], np.bincount(r[l, t], minlength=V)[:V]):
                        return f"one-hot tables (seed {seed})"
        for seed in range(4):
            b, table = wl.small_table_batch(seed, D=8, T_max=24)
            _, abs_sum = gather(b, table)
            if not np.array_equal(abs_sum, gather(b, table & np.uint16(0x7FFF))[0]):
                return f"sum of magnitudes (seed {seed})"
    return None


BATTERIES = {"index": index_pins_fail, "carry": carry_pins_fail, "embed": embed_pins_fail}


@pytest.mark.parametrize("kind", sorted(BATTERIES))
def test_unmutated_functions_pass_their_pins(workdir, kind):
    path = build_function_variant(workdir, f"clean_{kind}", "#include <stdint.h>",
                                  "#include <stdint.h>", "#include <stdint.h>")
    assert BATTERIES[kind](path) is None


@pytest.mark.parametrize("name", sorted(FUNCTION_MUTANTS))
def test_planted_mistake_in_index_carry_or_gather_is_caught(workdir, name):
    kind, anchor, old, new = FUNCTION_MUTANTS[name]
    path = build_function_variant(workdir, name, anchor, old, new)
    assert BATTERIES[kind](path) is not None, f"no pin catches the mutant {name}"
