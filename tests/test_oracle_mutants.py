"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a private copy of oracle/ple_oracle.c (a
dropped term, a wrong sign, an index off by one, a transposed operand, a
reversed order), compiles it with gcc into a temporary directory, and runs
the pin battery against it: the hand-worked window under both readings, the
sign/wrap cases, and the pure-Python brute force on random batches.  A
mutant that passes every pin would mean the pins leave that part of the
oracle unchecked, so each one must fail at least one pin.

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
