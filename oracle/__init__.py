"""CPU oracle for the PLE n-gram row-id hash -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or runs anything here, and this
package never imports the product path.

The arithmetic lives in ``ple_oracle.c`` (plain C, built with gcc); this
module only compiles it and marshals numpy arrays.  See that file's header
for the definition it follows: FreeToken PR #338, "perf(ple): fuse the n-gram
row-id hash into one Triton kernel", sections "What" and "Why it is safe".
"""

from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ple_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libple_oracle.so")

ORC_OK = 0
ORC_ERR_ARG = 1
ORC_ERR_GEOMETRY = 2
ORC_ERR_INDEX = 3
ORC_ERR_VOCAB = 4
ORC_ERR_ALLOC = 5

_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no GPU needed).  Returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
                    "-o", tmp, _SRC], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str) -> ctypes.CDLL:
    """A compiled copy of ple_oracle.c at `path`, with its C signatures."""
    lib = ctypes.CDLL(path)
    p, i32, i64, c_int = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int
    lib.oracle_floor_mod.argtypes = [i64, i64]
    lib.oracle_floor_mod.restype = i64
    lib.oracle_token_index.argtypes = [p, i32, i64, c_int, p, p]
    lib.oracle_token_index.restype = c_int
    lib.oracle_next_context.argtypes = [p, c_int, i64, p, p, p, i32, i32, p]
    lib.oracle_next_context.restype = c_int
    rargs = [p, c_int, i64, p, p, p, i32, i32, p, p, p, i32, i32, i32, i32, i64, p]
    lib.oracle_row_embed.argtypes = rargs[:-1] + [p, i64, i32, p, p]
    lib.oracle_row_embed.restype = c_int
    for name in ("oracle_row_ids", "oracle_row_ids_reading_b"):
        fn = getattr(lib, name)
        fn.argtypes = rargs
        fn.restype = c_int
    return lib


@contextlib.contextmanager
def using_library(path: str):
    """Route this module's functions through another compiled copy of the
    oracle (the tests' planted-mistake copies) for the duration."""
    global _lib
    lib = load_library(path)
    _load()
    with _lock:
        saved, _lib = _lib, lib
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a.size else None


def floor_mod(x: int, v: int) -> int:
    """torch.remainder semantics on int64 (floored; the divisor's sign)."""
    return int(_load().oracle_floor_mod(int(x), int(v)))


def token_index(cu_seqlens, num_requests: int, num_tokens: int, is_decode: bool):
    """(req, local) int32 arrays for a decode or a cu_seqlens-described prefill."""
    req = np.zeros(num_tokens, dtype=np.int32)
    local = np.zeros(num_tokens, dtype=np.int32)
    cu = None
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    rc = _load().oracle_token_index(_ptr(cu) if cu is not None else None, int(num_requests),
                                    int(num_tokens), int(bool(is_decode)), _ptr(req), _ptr(local))
    if rc != ORC_OK:
        raise OracleError(rc, "oracle_token_index")
    return req, local


def next_context(input_ids, req, local, ngram_context):
    """Each request's context for its next call: the last ctx_len ids of its
    context row followed by its tokens of this batch ([B, ctx_len])."""
    ids = np.ascontiguousarray(input_ids)
    ctx = np.ascontiguousarray(ngram_context, dtype=ids.dtype)
    req = np.ascontiguousarray(req, dtype=np.int32)
    local = np.ascontiguousarray(local, dtype=np.int32)
    out = np.zeros_like(ctx)
    rc = _load().oracle_next_context(_ptr(ids), ids.dtype.itemsize, ids.shape[0], _ptr(req),
                                     _ptr(local), _ptr(ctx), ctx.shape[0], ctx.shape[1],
                                     _ptr(out))
    if rc != ORC_OK:
        raise OracleError(rc, "oracle_next_context")
    return out


def row_ids(input_ids, req, local, ngram_context, layer_multipliers, vocab_sizes, offsets,
            ngram_size: int, heads_per_ngram: int, boundary_id: int, reading: str = "A"):
    """Row ids [L, T, H] int64 for one batch.

    ``layer_multipliers`` is [L, N] (or [N] for one layer), ``vocab_sizes``
    and ``offsets`` are [L, H] (or [H]); ``input_ids`` and ``ngram_context``
    share one dtype, int32 or int64.
    """
    ids = np.ascontiguousarray(input_ids)
    if ids.dtype not in (np.int32, np.int64):
        raise TypeError("input_ids must be int32 or int64")
    ctx = np.ascontiguousarray(ngram_context, dtype=ids.dtype)
    req = np.ascontiguousarray(req, dtype=np.int32)
    local = np.ascontiguousarray(local, dtype=np.int32)
    M = np.ascontiguousarray(layer_multipliers, dtype=np.int64)
    vocab = np.ascontiguousarray(vocab_sizes, dtype=np.int64)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    N = int(ngram_size)
    if M.ndim == 1:
        M = M.reshape(1, -1)
    if vocab.ndim == 1:
        vocab = vocab.reshape(1, -1)
    if off.ndim == 1:
        off = off.reshape(1, -1)
    L = M.shape[0]
    H = vocab.shape[1]
    T = ids.shape[0]
    if ctx.ndim == 1:
        ctx = ctx.reshape(-1, max(N - 1, 1))
    B = ctx.shape[0]
    ctx_len = ctx.shape[1] if ctx.ndim == 2 else 0
    if M.shape[1] != N or vocab.shape != (L, H) or off.shape != (L, H):
        raise ValueError("layer_multipliers must be [L, N]; vocab_sizes and offsets [L, H]")
    if req.shape != (T,) or local.shape != (T,):
        raise ValueError("req and local must be [T]")
    out = np.zeros((L, T, H), dtype=np.int64)
    fn = _load().oracle_row_ids if reading == "A" else _load().oracle_row_ids_reading_b
    rc = fn(_ptr(ids), ids.dtype.itemsize, T, _ptr(req), _ptr(local), _ptr(ctx), B, ctx_len,
            _ptr(M), _ptr(vocab), _ptr(off), H, N, int(heads_per_ngram), L, int(boundary_id),
            _ptr(out))
    if rc != ORC_OK:
        raise OracleError(rc, "oracle_row_ids")
    return out


def row_embed(input_ids, req, local, ngram_context, layer_multipliers, vocab_sizes, offsets,
              ngram_size: int, heads_per_ngram: int, boundary_id: int, table):
    """(emb, abs_sum), both [L, T, D] float64: the sum over heads of the rows
    of `table` ([L, V, D] bfloat16 bits as uint16) that the row ids name,
    and the sum of their absolute values (for an accumulation error bound).
    Row ids outside [0, V) add nothing."""
    ids = np.ascontiguousarray(input_ids)
    ctx = np.ascontiguousarray(ngram_context, dtype=ids.dtype)
    req = np.ascontiguousarray(req, dtype=np.int32)
    local = np.ascontiguousarray(local, dtype=np.int32)
    M = np.ascontiguousarray(layer_multipliers, dtype=np.int64).reshape(-1, int(ngram_size))
    L = M.shape[0]
    vocab = np.ascontiguousarray(vocab_sizes, dtype=np.int64).reshape(L, -1)
    off = np.ascontiguousarray(offsets, dtype=np.int64).reshape(L, -1)
    tab = np.ascontiguousarray(table, dtype=np.uint16)
    if tab.ndim != 3 or tab.shape[0] != L:
        raise ValueError("table must be [L, V, D]")
    T, H, V, D = ids.shape[0], vocab.shape[1], tab.shape[1], tab.shape[2]
    out = np.zeros((L, T, D), dtype=np.float64)
    abs_sum = np.zeros((L, T, D), dtype=np.float64)
    rc = _load().oracle_row_embed(_ptr(ids), ids.dtype.itemsize, T, _ptr(req), _ptr(local),
                                  _ptr(ctx), ctx.shape[0], ctx.shape[1], _ptr(M), _ptr(vocab),
                                  _ptr(off), H, int(ngram_size), int(heads_per_ngram), L,
                                  int(boundary_id), _ptr(tab), V, D, _ptr(out), _ptr(abs_sum))
    if rc != ORC_OK:
        raise OracleError(rc, "oracle_row_embed")
    return out, abs_sum
