"""Thin Python binding of libple.so (argument marshalling only).

Every function here checks and converts its arguments, then calls the C ABI
entry point of the same name; all computation happens in the library's CUDA
kernels on the tensors' device, on the current torch stream.  There is no CPU
path: tensors that are not all on one CUDA device are refused with
ValueError (FreeToken PR #338, "perf(ple): fuse the n-gram row-id hash into
one Triton kernel", section "Why it is safe": the fused path runs only when
every input is on the same CUDA device), and if the library is missing the
first call raises RuntimeError.

PyTorch is used only for device memory and streams.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

PLE_OK = 0
PLE_ERR_NULL = 1
PLE_ERR_SIZE = 2
PLE_ERR_GEOMETRY_CTX = 3
PLE_ERR_GEOMETRY_HEADS = 4
PLE_ERR_DTYPE = 5
PLE_ERR_ALIGN = 6
PLE_ERR_CUDA = 7
PLE_I32 = 0
PLE_I64 = 1
PLE_MAX_NGRAM = 16
PLE_MAX_HEADS = 256
PLE_MAX_EMBED_DIM = 65536
PLE_HEAD_BYTES = 48

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libple.so")

# every symbol include/ple.h declares, with its ctypes signature
_P, _I32, _I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
SIGNATURES = {
    "ple_build_token_index": (_I32, [_P, _I32, _I64, _I32, _P, _P, _P]),
    "ple_row_ids": (_I32, [_P, _I32, _I64, _P, _P, _P, _I32, _I32, _P, _P, _P, _I32, _I32, _I32,
                           _I32, _I64, _P, _P]),
    "ple_row_ids_i32": (_I32, [_P, _I32, _I64, _P, _P, _P, _I32, _I32, _P, _P, _P, _I32, _I32,
                               _I32, _I32, _I64, _P, _P]),
    "ple_row_ids_ex": (_I32, [_P, _I32, _I64, _P, _P, _P, _I32, _I32, _P, _P, _P, _I32, _I32,
                              _I32, _I32, _I64, _P, _I32, _P, _P, _P, _P]),
    "ple_prepare_heads": (_I32, [_P, _P, _I32, _I32, _P, _P]),
    "ple_row_embed": (_I32, [_P, _I32, _I64, _P, _P, _P, _I32, _I32, _P, _P, _P, _I32, _I32,
                             _I32, _I32, _I64, _P, _I64, _I32, _P, _P, _P, _P]),
    "ple_validate_index": (_I32, [_P, _I32, _I64, _I32, _P, _P, _P, _P]),
    "ple_selftest_floor_mod": (_I32, [_P, _P, _I64, _P, _P, _P]),
    "ple_status_string": (ctypes.c_char_p, [_I32]),
    "ple_last_cuda_error": (_I32, []),
    "ple_small_batch_max_rows": (_I64, []),
    "ple_set_programmatic_launch": (_I32, [_I32]),
    "ple_shard_plan": (_I32, [_P, _I32, _I64, _I32, _I32, _P, _P, _P, _P]),
    "ple_shard_inputs": (_I32, [_P, _I32, _P, _P, _I32, _I64, _I32, _I64, _I64, _I32, _I32, _P,
                                _P, _P]),
}

_lock = threading.Lock()
_lib = None


class PleError(RuntimeError):
    """A non-geometry failure reported by the library."""

    def __init__(self, status: int, where: str):
        msg = status_string(status)
        if status == PLE_ERR_CUDA:
            msg += f" (cudaError {lib().ple_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded libple.so.  Raises RuntimeError if it was never built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"libple.so is not built ({LIB_PATH}); build it with "
                        "layer_gram_embedding_gb300.build.build() -- there is no fallback path")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().ple_status_string(int(status)).decode()


def small_batch_max_rows() -> int:
    """Batches of at most this many row ids (T * H * L) run the small-batch
    kernel; the row ids do not depend on which kernel runs."""
    return int(lib().ple_small_batch_max_rows())


def set_programmatic_launch(enabled: bool) -> bool:
    """Turn programmatic dependent launch of every library kernel on or off
    (process-wide; on by default); returns the previous setting.  Off, each
    call is an ordinary stream-ordered launch, so one call's device time
    stands alone; the row ids are the same either way."""
    return bool(lib().ple_set_programmatic_launch(1 if enabled else 0))


def _check(status: int, where: str):
    if status == PLE_OK:
        return
    if status in (PLE_ERR_GEOMETRY_CTX, PLE_ERR_GEOMETRY_HEADS):
        raise ValueError(f"{where}: {status_string(status)}")
    raise PleError(status, where)


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else ctypes.c_void_p(0)


def _one_cuda_device(tensors, where: str) -> torch.device:
    devs = {t.device for t in tensors if t is not None}
    if len(devs) != 1 or next(iter(devs)).type != "cuda":
        raise ValueError(f"{where}: every tensor must be on one CUDA device (got {sorted(map(str, devs))})")
    return next(iter(devs))


def _need(t: torch.Tensor, dtype, name: str, where: str):
    if t.dtype != dtype:
        raise TypeError(f"{where}: {name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{where}: {name} must be contiguous")


def ple_build_token_index(cu_seqlens, num_requests: int, num_tokens: int, is_decode: bool,
                          req: torch.Tensor | None = None, local: torch.Tensor | None = None,
                          device=None, stream=None):
    """(req, local) int32 [T] for a decode (is_decode) or a cu_seqlens prefill.

    cu_seqlens: int32 [num_requests + 1] CUDA tensor (ignored for a decode).
    req / local: optional preallocated int32 [T] outputs (e.g. graph buffers).
    """
    where = "ple_build_token_index"
    T = int(num_tokens)
    tensors = [t for t in (cu_seqlens if not is_decode else None, req, local) if t is not None]
    if device is None and not tensors:
        raise ValueError(f"{where}: pass a device, cu_seqlens or the output buffers")
    dev = torch.device(device) if device is not None else _one_cuda_device(tensors, where)
    if tensors:
        _one_cuda_device(tensors + [torch.empty(0, device=dev)], where)
    if req is None:
        req = torch.empty(T, dtype=torch.int32, device=dev)
    if local is None:
        local = torch.empty(T, dtype=torch.int32, device=dev)
    for name, t in (("req", req), ("local", local)):
        _need(t, torch.int32, name, where)
        if t.numel() != T:
            raise ValueError(f"{where}: {name} must have num_tokens elements")
    cu_p = ctypes.c_void_p(0)
    if not is_decode:
        _need(cu_seqlens, torch.int32, "cu_seqlens", where)
        if cu_seqlens.numel() != int(num_requests) + 1:
            raise ValueError(f"{where}: cu_seqlens must have num_requests + 1 elements")
        cu_p = _ptr(cu_seqlens)
    with torch.cuda.device(dev):
        st = lib().ple_build_token_index(cu_p, int(num_requests), T, int(bool(is_decode)),
                                         _ptr(req), _ptr(local), _stream_handle(stream, dev))
    _check(st, where)
    return req, local


def ple_shard_plan(cu_seqlens, num_requests: int, num_tokens: int, world_size: int,
                   rank: int):
    """(token_begin, token_end, request_begin, request_count) of one rank's
    share of a batch split by token range -- host code on a host int32
    cu_seqlens [num_requests + 1] (numpy array or CPU tensor), or None for a
    decode batch.  Needs no GPU."""
    where = "ple_shard_plan"
    cu_p = ctypes.c_void_p(0)
    keep = None
    if cu_seqlens is not None:
        keep = torch.as_tensor(cu_seqlens)
        if keep.device.type != "cpu" or keep.dtype != torch.int32:
            raise ValueError(f"{where}: cu_seqlens must be a host int32 array")
        keep = keep.contiguous()
        if keep.numel() != int(num_requests) + 1:
            raise ValueError(f"{where}: cu_seqlens must have num_requests + 1 elements")
        cu_p = ctypes.c_void_p(keep.data_ptr())
    tb, te = ctypes.c_int64(), ctypes.c_int64()
    rb, rc = ctypes.c_int32(), ctypes.c_int32()
    st = lib().ple_shard_plan(cu_p, int(num_requests), int(num_tokens), int(world_size),
                              int(rank), ctypes.byref(tb), ctypes.byref(te), ctypes.byref(rb),
                              ctypes.byref(rc))
    _check(st, where)
    del keep
    return tb.value, te.value, rb.value, rc.value


def ple_shard_inputs(input_ids: torch.Tensor, cu_seqlens: torch.Tensor,
                     ngram_context: torch.Tensor, plan, shard_cu_seqlens=None,
                     shard_context=None, stream=None):
    """One rank's (ids, cu_seqlens, ngram_context) for its plan from
    ple_shard_plan, built on the device from the whole batch's device
    tensors (one launch).  The ids are a view of input_ids; the other two are
    written into shard_cu_seqlens [request_count + 1] int32 and shard_context
    [request_count, ngram_size - 1] (allocated when None)."""
    where = "ple_shard_inputs"
    tb, te, rb, rc = (int(x) for x in plan)
    dev = _one_cuda_device([input_ids, cu_seqlens, ngram_context], where)
    if input_ids.dtype not in (torch.int32, torch.int64) or ngram_context.dtype != input_ids.dtype:
        raise ValueError(f"{where}: ids and context must be int32 or int64, same dtype")
    _need(cu_seqlens, torch.int32, "cu_seqlens", where)
    if ngram_context.dim() != 2:
        raise ValueError(f"{where}: ngram_context must be [B, ngram_size - 1]")
    B, C = ngram_context.shape
    if cu_seqlens.numel() != B + 1:
        raise ValueError(f"{where}: cu_seqlens must have num_requests + 1 elements")
    if not 0 <= tb < te <= input_ids.numel() or rb < 0 or rc < 1 or rb + rc > B:
        raise ValueError(f"{where}: the plan does not fit this batch (or the share is empty)")
    if shard_cu_seqlens is None:
        shard_cu_seqlens = torch.empty(max(rc, 0) + 1, dtype=torch.int32, device=dev)
    if shard_context is None:
        shard_context = torch.empty((max(rc, 0), C), dtype=input_ids.dtype, device=dev)
    _one_cuda_device([input_ids, shard_cu_seqlens, shard_context], where)
    if shard_cu_seqlens.numel() != rc + 1 or tuple(shard_context.shape) != (rc, C):
        raise ValueError(f"{where}: outputs must be [request_count + 1] and [request_count, C]")
    for name, t in (("input_ids", input_ids), ("cu_seqlens", cu_seqlens),
                    ("ngram_context", ngram_context), ("shard_cu_seqlens", shard_cu_seqlens),
                    ("shard_context", shard_context)):
        if not t.is_contiguous():
            raise ValueError(f"{where}: {name} must be contiguous")
    dt = PLE_I32 if input_ids.dtype == torch.int32 else PLE_I64
    with torch.cuda.device(dev):
        st = lib().ple_shard_inputs(_ptr(input_ids), dt, _ptr(cu_seqlens), _ptr(ngram_context),
                                    int(B), int(input_ids.numel()), int(C), tb, te, rb, rc,
                                    _ptr(shard_cu_seqlens), _ptr(shard_context),
                                    _stream_handle(stream, dev))
    _check(st, where)
    return input_ids[tb:te], shard_cu_seqlens, shard_context


def ple_row_ids(input_ids: torch.Tensor, req: torch.Tensor | None, local: torch.Tensor | None,
                ngram_context: torch.Tensor, layer_multipliers: torch.Tensor,
                vocab_sizes: torch.Tensor, offsets: torch.Tensor, ngram_size: int,
                heads_per_ngram: int, boundary_id: int, out: torch.Tensor | None = None,
                stream=None, out_dtype=torch.int64, cu_seqlens: torch.Tensor | None = None,
                next_context: torch.Tensor | None = None,
                heads: torch.Tensor | None = None) -> torch.Tensor:
    """Row ids [L, T, H] int64 (one launch for every layer).

    out_dtype=torch.int32 calls ple_row_ids_i32 instead: the low 32 bits of
    each row id, half the output bytes.  next_context ([B, ngram_size-1],
    dtype of the ids, not overlapping ngram_context) receives each request's
    carried context in the same launch (ple_row_ids_ex); with req and local
    it needs cu_seqlens.  req = local = None with cu_seqlens ([B+1] int32):
    the kernel finds each token's request by searching cu_seqlens, so no
    index is built or read.  heads: the constants ple_prepare_heads made from
    these vocab_sizes and offsets, read instead of deriving them in the call
    (ple_row_ids_ex).

    input_ids [T] and ngram_context [B, ngram_size-1]: int32 or int64, same
    dtype.  layer_multipliers [L, N] (or [N]), vocab_sizes and offsets
    [L, H] (or [H]): int64.  out: optional fixed [L, T, H] int64 destination
    (a graph replay then writes into a stable buffer).  req and local both
    None: a decode batch (one token per request at offset 0, B == T), with no
    index to build or read (without cu_seqlens).  ValueError on the two
    geometry preconditions and on tensors not all on one CUDA device.
    """
    where = "ple_row_ids"
    if (req is None) != (local is None):
        raise ValueError(f"{where}: pass both req and local, or neither (decode)")
    dev = _one_cuda_device([t for t in (input_ids, req, local, ngram_context, layer_multipliers,
                                        vocab_sizes, offsets, out, cu_seqlens, next_context,
                                        heads) if t is not None], where)
    if input_ids.dtype not in (torch.int32, torch.int64):
        raise TypeError(f"{where}: input_ids must be int32 or int64")
    if ngram_context.dtype != input_ids.dtype:
        raise TypeError(f"{where}: ngram_context must have the dtype of input_ids")
    if input_ids.dim() != 1:
        raise ValueError(f"{where}: input_ids must be [T]")
    T = input_ids.shape[0]
    N = int(ngram_size)
    M = layer_multipliers.reshape(1, -1) if layer_multipliers.dim() == 1 else layer_multipliers
    vocab = vocab_sizes.reshape(1, -1) if vocab_sizes.dim() == 1 else vocab_sizes
    off = offsets.reshape(1, -1) if offsets.dim() == 1 else offsets
    L, H = vocab.shape[0], vocab.shape[1]
    ctx = ngram_context
    if ctx.dim() != 2:
        raise ValueError(f"{where}: ngram_context must be [B, ctx_len]")
    for name, t in (("input_ids", input_ids), ("ngram_context", ctx)):
        if not t.is_contiguous():
            raise ValueError(f"{where}: {name} must be contiguous")
    if req is not None:
        for name, t in (("req", req), ("local", local)):
            _need(t, torch.int32, name, where)
            if t.numel() != T:
                raise ValueError(f"{where}: {name} must be [T]")
    for name, t in (("layer_multipliers", M), ("vocab_sizes", vocab), ("offsets", off)):
        _need(t, torch.int64, name, where)
    if M.shape != (L, N):
        raise ValueError(f"{where}: layer_multipliers must be [L, ngram_size]")
    if off.shape != (L, H):
        raise ValueError(f"{where}: offsets must have the shape of vocab_sizes")
    if out_dtype not in (torch.int64, torch.int32):
        raise TypeError(f"{where}: out_dtype must be torch.int64 or torch.int32")
    if heads is not None:
        _need(heads, torch.uint8, "heads", where)
        if tuple(heads.shape) != (L, H, PLE_HEAD_BYTES) or heads.device != dev:
            raise ValueError(f"{where}: heads must be ple_prepare_heads' [L, H, "
                             f"{PLE_HEAD_BYTES}] on the ids' device")
    if out is None:
        out = torch.empty((L, T, H), dtype=out_dtype, device=dev)
    else:
        _need(out, out_dtype, "out", where)
        if tuple(out.shape) not in ((L, T, H),) + (((T, H),) if L == 1 else ()):
            raise ValueError(f"{where}: out must be [L, T, H]")
    dtype_code = PLE_I64 if input_ids.dtype == torch.int64 else PLE_I32
    with torch.cuda.device(dev):
        common = (_ptr(input_ids), dtype_code, T,
                  _ptr(req) if req is not None else ctypes.c_void_p(0),
                  _ptr(local) if local is not None else ctypes.c_void_p(0), _ptr(ctx),
                  ctx.shape[0], ctx.shape[1], _ptr(M), _ptr(vocab), _ptr(off), H, N,
                  int(heads_per_ngram), L, int(boundary_id), _ptr(out))
        # cu_seqlens matters to the kernel for the carry and for the search
        # mode (no index); otherwise it is not passed
        use_cu = cu_seqlens is not None and (next_context is not None or req is None)
        if next_context is None and heads is None and not use_cu:
            fn = lib().ple_row_ids if out_dtype == torch.int64 else lib().ple_row_ids_i32
            st = fn(*common, _stream_handle(stream, dev))
        else:
            null = ctypes.c_void_p(0)
            if next_context is not None:
                if (next_context.dtype != input_ids.dtype
                        or tuple(next_context.shape) != tuple(ctx.shape)):
                    raise ValueError(
                        f"{where}: next_context must be [B, ngram_size-1] of the ids' dtype")
                if not next_context.is_contiguous() or next_context.device != dev:
                    raise ValueError(
                        f"{where}: next_context must be contiguous, on the ids' device")
            if use_cu:
                _need(cu_seqlens, torch.int32, "cu_seqlens", where)
                if cu_seqlens.device != dev or cu_seqlens.numel() != ctx.shape[0] + 1:
                    raise ValueError(f"{where}: cu_seqlens must be [B + 1] on the ids' device")
            st = lib().ple_row_ids_ex(*common, PLE_I64 if out_dtype == torch.int64 else PLE_I32,
                                      _ptr(cu_seqlens) if use_cu else null,
                                      _ptr(next_context) if next_context is not None else null,
                                      _ptr(heads) if heads is not None else null,
                                      _stream_handle(stream, dev))
    _check(st, where)
    return out


def ple_prepare_heads(vocab_sizes: torch.Tensor, offsets: torch.Tensor,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """[L, H, PLE_HEAD_BYTES] uint8: each head's remainder constants, set up
    once for these vocab_sizes and offsets ([L, H] or [H] int64 on a CUDA
    device) and passed to ple_row_ids(heads=...) call after call."""
    where = "ple_prepare_heads"
    dev = _one_cuda_device([t for t in (vocab_sizes, offsets, out) if t is not None], where)
    vocab = vocab_sizes.reshape(1, -1) if vocab_sizes.dim() == 1 else vocab_sizes
    off = offsets.reshape(1, -1) if offsets.dim() == 1 else offsets
    for name, t in (("vocab_sizes", vocab), ("offsets", off)):
        _need(t, torch.int64, name, where)
    if off.shape != vocab.shape or vocab.dim() != 2:
        raise ValueError(f"{where}: vocab_sizes and offsets must be [L, H]")
    L, H = vocab.shape
    if out is None:
        out = torch.empty((L, H, PLE_HEAD_BYTES), dtype=torch.uint8, device=dev)
    else:
        _need(out, torch.uint8, "out", where)
        if tuple(out.shape) != (L, H, PLE_HEAD_BYTES):
            raise ValueError(f"{where}: out must be [L, H, {PLE_HEAD_BYTES}]")
    with torch.cuda.device(dev):
        st = lib().ple_prepare_heads(_ptr(vocab), _ptr(off), L, H, _ptr(out),
                                     _stream_handle(stream, dev))
    _check(st, where)
    return out


def ple_row_embed(input_ids: torch.Tensor, req: torch.Tensor | None, local: torch.Tensor | None,
                  ngram_context: torch.Tensor, layer_multipliers: torch.Tensor,
                  vocab_sizes: torch.Tensor, offsets: torch.Tensor, ngram_size: int,
                  heads_per_ngram: int, boundary_id: int, table: torch.Tensor,
                  out: torch.Tensor | None = None, stream=None,
                  cu_seqlens: torch.Tensor | None = None,
                  heads: torch.Tensor | None = None) -> torch.Tensor:
    """[L, T, D] float32: per layer and token, the sum over heads of the rows
    of `table` ([L, V, D] bfloat16, or its raw 16-bit patterns) that the row
    ids name -- the hash and the gather in one launch, the row ids never
    written.  Other arguments as ple_row_ids (req = local = None with
    cu_seqlens: the requests found in the kernel; heads: prepared
    constants)."""
    where = "ple_row_embed"
    if (req is None) != (local is None):
        raise ValueError(f"{where}: pass both req and local, or neither (decode)")
    dev = _one_cuda_device([t for t in (input_ids, req, local, ngram_context, layer_multipliers,
                                        vocab_sizes, offsets, table, out, cu_seqlens, heads)
                            if t is not None], where)
    if table.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"{where}: table must be bfloat16 (or its 16-bit patterns)")
    if table.dim() != 3 or not table.is_contiguous():
        raise ValueError(f"{where}: table must be a contiguous [L, V, D] tensor")
    M = layer_multipliers.reshape(1, -1) if layer_multipliers.dim() == 1 else layer_multipliers
    vocab = vocab_sizes.reshape(1, -1) if vocab_sizes.dim() == 1 else vocab_sizes
    off = offsets.reshape(1, -1) if offsets.dim() == 1 else offsets
    for name, t in (("layer_multipliers", M), ("vocab_sizes", vocab), ("offsets", off)):
        _need(t, torch.int64, name, where)
    L, H = vocab.shape
    T = input_ids.shape[0]
    V, D = table.shape[1], table.shape[2]
    if table.shape[0] != L or M.shape != (L, int(ngram_size)) or off.shape != (L, H):
        raise ValueError(f"{where}: table [L, V, D], layer_multipliers [L, N], offsets [L, H]")
    if input_ids.dtype not in (torch.int32, torch.int64) or ngram_context.dtype != input_ids.dtype:
        raise TypeError(f"{where}: input_ids and ngram_context must share int32 or int64")
    if req is not None:
        for name, t in (("req", req), ("local", local)):
            _need(t, torch.int32, name, where)
    if out is None:
        out = torch.empty((L, T, D), dtype=torch.float32, device=dev)
    else:
        _need(out, torch.float32, "out", where)
        if tuple(out.shape) != (L, T, D):
            raise ValueError(f"{where}: out must be [L, T, D]")
    ctx = ngram_context
    use_cu = cu_seqlens is not None and req is None
    if use_cu:
        _need(cu_seqlens, torch.int32, "cu_seqlens", where)
        if cu_seqlens.numel() != ctx.shape[0] + 1:
            raise ValueError(f"{where}: cu_seqlens must be [B + 1]")
    if heads is not None:
        _need(heads, torch.uint8, "heads", where)
        if tuple(heads.shape) != (L, H, PLE_HEAD_BYTES):
            raise ValueError(f"{where}: heads must be ple_prepare_heads' [L, H, "
                             f"{PLE_HEAD_BYTES}]")
    with torch.cuda.device(dev):
        st = lib().ple_row_embed(
            _ptr(input_ids), PLE_I64 if input_ids.dtype == torch.int64 else PLE_I32, T,
            _ptr(req) if req is not None else ctypes.c_void_p(0),
            _ptr(local) if local is not None else ctypes.c_void_p(0), _ptr(ctx), ctx.shape[0],
            ctx.shape[1], _ptr(M), _ptr(vocab), _ptr(off), H, int(ngram_size),
            int(heads_per_ngram), L, int(boundary_id), _ptr(table), V, D, _ptr(out),
            _ptr(cu_seqlens) if use_cu else ctypes.c_void_p(0),
            _ptr(heads) if heads is not None else ctypes.c_void_p(0),
            _stream_handle(stream, dev))
    _check(st, where)
    return out


def ple_validate_index(cu_seqlens, num_requests: int, num_tokens: int, is_decode: bool,
                       req: torch.Tensor, local: torch.Tensor, stream=None) -> torch.Tensor:
    """A one-element int64 CUDA tensor: the first token whose (req, local)
    is not what cu_seqlens (or the decode rule) defines, or num_tokens when
    every token is right.  Asynchronous: read it when the stream has run."""
    where = "ple_validate_index"
    dev = _one_cuda_device([t for t in (cu_seqlens if not is_decode else None, req, local)
                            if t is not None], where)
    for name, t in (("req", req), ("local", local)):
        _need(t, torch.int32, name, where)
    first_bad = torch.full((1,), int(num_tokens), dtype=torch.int64, device=dev)
    cu_p = ctypes.c_void_p(0)
    if not is_decode:
        _need(cu_seqlens, torch.int32, "cu_seqlens", where)
        cu_p = _ptr(cu_seqlens)
    with torch.cuda.device(dev):
        st = lib().ple_validate_index(cu_p, int(num_requests), int(num_tokens),
                                      int(bool(is_decode)), _ptr(req), _ptr(local),
                                      _ptr(first_bad), _stream_handle(stream, dev))
    _check(st, where)
    return first_bad


def ple_selftest_floor_mod(x: torch.Tensor, v: torch.Tensor, stream=None):
    """(library floored remainder, CUDA % with sign fix), elementwise."""
    where = "ple_selftest_floor_mod"
    dev = _one_cuda_device([x, v], where)
    _need(x, torch.int64, "x", where)
    _need(v, torch.int64, "v", where)
    if x.shape != v.shape:
        raise ValueError(f"{where}: x and v must have one shape")
    fast = torch.empty_like(x)
    ref = torch.empty_like(x)
    with torch.cuda.device(dev):
        st = lib().ple_selftest_floor_mod(_ptr(x), _ptr(v), x.numel(), _ptr(fast), _ptr(ref),
                                          _stream_handle(stream, dev))
    _check(st, where)
    return fast, ref
