"""The C ABI without a GPU: the library builds, loads, exports every symbol
include/ple.h declares, and its host-side argument checks return the right
status before anything touches CUDA.  No call here reaches a launch."""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

import layer_gram_embedding_gb300 as ple
from layer_gram_embedding_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "ple.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ple.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ple_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_are_all_exported(lib):
    names = declared_functions()
    assert names == sorted(binding.SIGNATURES), names
    for n in names:
        assert getattr(lib, n) is not None


def test_header_constants_match_binding():
    text = open(HEADER).read()
    consts = dict(re.findall(r"(PLE_[A-Z_0-9]+)\s*=\s*(\d+)", text))
    consts.update(dict(re.findall(r"#define\s+(PLE_[A-Z_]+)\s+(\d+)", text)))
    for k, v in consts.items():
        assert getattr(binding, k) == int(v), k


def test_status_strings(lib):
    for s in range(8):
        assert ple.status_string(s) and ple.status_string(s) != "unknown status"
    assert ple.status_string(99) == "unknown status"
    assert lib.ple_last_cuda_error() == 0


def test_programmatic_launch_switch(lib):
    # host-side only: the switch is process-wide and returns the previous value
    assert ple.set_programmatic_launch(False) is True
    assert ple.set_programmatic_launch(False) is False
    assert ple.set_programmatic_launch(True) is False
    assert lib.ple_set_programmatic_launch(7) == 1
    assert lib.ple_set_programmatic_launch(1) == 1


# fake, never dereferenced device addresses: every call below fails a host
# check before the library touches CUDA
A = 0x10000
MIS = 0x10001


def row_ids(lib, **kw):
    a = dict(ids=A, dtype=1, T=64, req=A, local=A, ctx=A, B=1, ctx_len=2, M=A, vocab=A, off=A,
             H=4, N=3, hpn=2, L=1, b=7, out=A)
    a.update(kw)
    return lib.ple_row_ids(a["ids"], a["dtype"], a["T"], a["req"], a["local"], a["ctx"], a["B"],
                           a["ctx_len"], a["M"], a["vocab"], a["off"], a["H"], a["N"], a["hpn"],
                           a["L"], a["b"], a["out"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(N=1, ctx_len=0, H=0), ple.PLE_ERR_SIZE),
    (dict(N=17, ctx_len=16, H=32), ple.PLE_ERR_SIZE),
    (dict(hpn=0, H=0), ple.PLE_ERR_SIZE),
    (dict(L=0), ple.PLE_ERR_SIZE),
    (dict(T=-1), ple.PLE_ERR_SIZE),
    (dict(T=2 ** 31), ple.PLE_ERR_SIZE),
    (dict(T=2 ** 30, L=2 ** 30), ple.PLE_ERR_SIZE),          # L*T*H*8 bytes overflow int64
    (dict(T=2 ** 28, L=2 ** 28, out=A + 4), ple.PLE_ERR_ALIGN),  # 2^61 bytes: past the size check
    (dict(ctx_len=3), ple.PLE_ERR_GEOMETRY_CTX),
    (dict(ctx_len=1), ple.PLE_ERR_GEOMETRY_CTX),
    (dict(H=5), ple.PLE_ERR_GEOMETRY_HEADS),
    (dict(hpn=1), ple.PLE_ERR_GEOMETRY_HEADS),
    (dict(hpn=200, H=400), ple.PLE_ERR_SIZE),
    (dict(B=0), ple.PLE_ERR_SIZE),
    (dict(ids=None), ple.PLE_ERR_NULL),
    (dict(req=None), ple.PLE_ERR_NULL),
    (dict(local=None), ple.PLE_ERR_NULL),
    (dict(req=None, local=None), ple.PLE_ERR_SIZE),          # index-free needs B == T
    (dict(req=None, local=None, T=4, B=5), ple.PLE_ERR_SIZE),
    (dict(ctx=None), ple.PLE_ERR_NULL),
    (dict(M=None), ple.PLE_ERR_NULL),
    (dict(vocab=None), ple.PLE_ERR_NULL),
    (dict(off=None), ple.PLE_ERR_NULL),
    (dict(out=None), ple.PLE_ERR_NULL),
    (dict(dtype=2), ple.PLE_ERR_DTYPE),
    (dict(ids=A + 4), ple.PLE_ERR_ALIGN),
    (dict(ids=A + 4, dtype=0, ctx=A + 2), ple.PLE_ERR_ALIGN),
    (dict(req=A + 2), ple.PLE_ERR_ALIGN),
    (dict(out=A + 4), ple.PLE_ERR_ALIGN),
    (dict(vocab=MIS), ple.PLE_ERR_ALIGN),
])
def test_row_ids_host_checks(lib, kw, status):
    assert row_ids(lib, **kw) == status


def row_ids_ex(lib, **kw):
    a = dict(ids=A, dtype=1, T=64, req=A, local=A, ctx=A, B=1, ctx_len=2, M=A, vocab=A, off=A,
             H=4, N=3, hpn=2, L=1, b=7, out=A, out_dtype=1, cu=A, nxt=A, heads=None)
    a.update(kw)
    return lib.ple_row_ids_ex(a["ids"], a["dtype"], a["T"], a["req"], a["local"], a["ctx"],
                              a["B"], a["ctx_len"], a["M"], a["vocab"], a["off"], a["H"], a["N"],
                              a["hpn"], a["L"], a["b"], a["out"], a["out_dtype"], a["cu"],
                              a["nxt"], a["heads"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(out_dtype=2), ple.PLE_ERR_DTYPE),
    (dict(out_dtype=2, ctx_len=1), ple.PLE_ERR_GEOMETRY_CTX),   # geometry first
    (dict(out_dtype=-1, T=0), ple.PLE_ERR_DTYPE),
    (dict(cu=None), ple.PLE_ERR_NULL),                          # carry needs cu_seqlens
    (dict(nxt=A + 4), ple.PLE_ERR_ALIGN),
    (dict(cu=A + 2), ple.PLE_ERR_ALIGN),
    (dict(out_dtype=0, out=A + 2), ple.PLE_ERR_ALIGN),
    (dict(out_dtype=1, out=A + 4), ple.PLE_ERR_ALIGN),
    (dict(req=None, local=None, cu=None, T=4, B=5), ple.PLE_ERR_SIZE),
    (dict(heads=A + 8), ple.PLE_ERR_ALIGN),                     # prepared constants: 16 bytes
    (dict(vocab=None, off=None, out_dtype=2), ple.PLE_ERR_NULL),
    # with prepared constants vocab_sizes and offsets are not needed: the
    # call gets past the pointer checks to the output dtype
    (dict(vocab=None, off=None, heads=A, out_dtype=2), ple.PLE_ERR_DTYPE),
    (dict(vocab=None, off=None, heads=A, ids=None), ple.PLE_ERR_NULL),
    # req = local = NULL with cu_seqlens: the kernel searches cu_seqlens, so
    # B != T is accepted (the call gets past the index checks to out_dtype)
    (dict(req=None, local=None, T=4, B=5, out_dtype=2), ple.PLE_ERR_DTYPE),
    (dict(req=None, local=None, T=4, B=5, cu=A + 2), ple.PLE_ERR_ALIGN),
    (dict(cu=A + 2, nxt=None), ple.PLE_ERR_ALIGN),
])
def test_row_ids_ex_host_checks(lib, kw, status):
    assert row_ids_ex(lib, **kw) == status


@pytest.mark.parametrize("args,status", [
    ((A, A, 0, 4, A), ple.PLE_ERR_SIZE),
    ((A, A, 1, 0, A), ple.PLE_ERR_SIZE),
    ((A, A, 1, 257, A), ple.PLE_ERR_SIZE),
    ((None, A, 1, 4, A), ple.PLE_ERR_NULL),
    ((A, None, 1, 4, A), ple.PLE_ERR_NULL),
    ((A, A, 1, 4, None), ple.PLE_ERR_NULL),
    ((MIS, A, 1, 4, A), ple.PLE_ERR_ALIGN),
    ((A, A, 1, 4, A + 8), ple.PLE_ERR_ALIGN),
])
def test_prepare_heads_host_checks(lib, args, status):
    assert lib.ple_prepare_heads(*args, None) == status


def row_embed(lib, **kw):
    a = dict(ids=A, dtype=1, T=64, req=A, local=A, ctx=A, B=1, ctx_len=2, M=A, vocab=A, off=A,
             H=4, N=3, hpn=2, L=1, b=7, table=A, V=100, D=64, out=A, cu=None, heads=None)
    a.update(kw)
    return lib.ple_row_embed(a["ids"], a["dtype"], a["T"], a["req"], a["local"], a["ctx"],
                             a["B"], a["ctx_len"], a["M"], a["vocab"], a["off"], a["H"], a["N"],
                             a["hpn"], a["L"], a["b"], a["table"], a["V"], a["D"], a["out"],
                             a["cu"], a["heads"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(ctx_len=1), ple.PLE_ERR_GEOMETRY_CTX),
    (dict(D=4), ple.PLE_ERR_SIZE),
    (dict(D=12), ple.PLE_ERR_SIZE),
    (dict(D=65544), ple.PLE_ERR_SIZE),
    (dict(V=-1), ple.PLE_ERR_SIZE),
    (dict(V=2 ** 62), ple.PLE_ERR_SIZE),
    (dict(T=2 ** 25, L=2 ** 25, D=65536, V=16), ple.PLE_ERR_SIZE),  # L*T*dim*4 bytes overflow
    (dict(T=2 ** 22, L=2 ** 22, D=65536, V=16, out=A + 4), ple.PLE_ERR_ALIGN),  # 2^62 bytes fit
    (dict(table=None), ple.PLE_ERR_NULL),
    (dict(out=None), ple.PLE_ERR_NULL),
    (dict(table=A + 8), ple.PLE_ERR_ALIGN),
    (dict(out=A + 4), ple.PLE_ERR_ALIGN),
    (dict(T=0, table=None, out=None), ple.PLE_OK),
    (dict(heads=A + 8), ple.PLE_ERR_ALIGN),
    (dict(req=None, local=None, T=4, B=5, cu=A + 2), ple.PLE_ERR_ALIGN),
    # with cu_seqlens B != T is accepted: the call gets past the index checks
    (dict(req=None, local=None, T=4, B=5, cu=A, table=A + 8), ple.PLE_ERR_ALIGN),
    (dict(req=None, local=None, T=4, B=5), ple.PLE_ERR_SIZE),          # decode needs B == T
    (dict(vocab=None, off=None, heads=A, D=12), ple.PLE_ERR_SIZE),     # past the NULL checks
])
def test_row_embed_host_checks(lib, kw, status):
    assert row_embed(lib, **kw) == status


def test_row_ids_empty_batch_is_ok_without_pointers(lib):
    assert row_ids(lib, T=0, ids=None, req=None, local=None, ctx=None, M=None, vocab=None,
                   off=None, out=None, B=0) == ple.PLE_OK


def test_geometry_is_checked_before_emptiness(lib):
    # the two preconditions are refused even for an empty batch
    assert row_ids(lib, T=0, ctx_len=5) == ple.PLE_ERR_GEOMETRY_CTX


@pytest.mark.parametrize("args,status", [
    ((A, 2, -1, 0, A, A), ple.PLE_ERR_SIZE),
    ((A, 0, 5, 0, A, A), ple.PLE_ERR_SIZE),
    ((None, 3, 5, 1, A, A), ple.PLE_ERR_SIZE),      # decode needs B == T
    ((None, 2, 5, 0, A, A), ple.PLE_ERR_NULL),      # prefill needs cu_seqlens
    ((A, 2, 5, 0, None, A), ple.PLE_ERR_NULL),
    ((A, 2, 5, 0, A, None), ple.PLE_ERR_NULL),
    ((MIS, 2, 5, 0, A, A), ple.PLE_ERR_ALIGN),
    ((A, 2, 5, 0, A + 2, A), ple.PLE_ERR_ALIGN),
    ((None, 0, 0, 0, None, None), ple.PLE_OK),      # T == 0: nothing to do
])
def test_token_index_host_checks(lib, args, status):
    assert lib.ple_build_token_index(*args, None) == status


def test_selftest_host_checks(lib):
    assert lib.ple_selftest_floor_mod(A, A, -1, A, A, None) == ple.PLE_ERR_SIZE
    assert lib.ple_selftest_floor_mod(None, None, 0, None, None, None) == ple.PLE_OK
    assert lib.ple_selftest_floor_mod(None, A, 4, A, A, None) == ple.PLE_ERR_NULL
    assert lib.ple_selftest_floor_mod(A, A, 4, A, MIS, None) == ple.PLE_ERR_ALIGN


def test_binding_refuses_cpu_tensors():
    # the fused path is only for CUDA tensors; there is no CPU fallback
    z64 = torch.zeros(4, dtype=torch.int64)
    z32 = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        ple.ple_row_ids(z64, z32, z32, torch.zeros((1, 2), dtype=torch.int64),
                        torch.zeros((1, 3), dtype=torch.int64), torch.ones((1, 4), dtype=torch.int64),
                        torch.zeros((1, 4), dtype=torch.int64), 3, 2, 7)
    with pytest.raises(ValueError, match="CUDA"):
        ple.ple_build_token_index(torch.tensor([0, 4], dtype=torch.int32), 1, 4, False)


def test_library_has_no_host_compute_path():
    # the package never imports the oracle, and the oracle never imports it
    pkg = os.path.dirname(ple.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(root, f)).read()
                assert "oracle" not in src.replace("the oracle", ""), f
    ora = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")
    for f in os.listdir(ora):
        if f.endswith((".py", ".c")):
            assert "layer_gram_embedding_gb300" not in open(os.path.join(ora, f)).read()


def test_bench_kernel_source_list_exists():
    import bench
    assert len(bench.kernel_source_hash()) == 16


@pytest.mark.parametrize("args,status", [
    ((A, 2, -1, 0, A, A, A), ple.PLE_ERR_SIZE),
    ((A, 0, 5, 0, A, A, A), ple.PLE_ERR_SIZE),
    ((None, 3, 5, 1, A, A, A), ple.PLE_ERR_SIZE),
    ((None, 2, 5, 0, A, A, A), ple.PLE_ERR_NULL),
    ((A, 2, 5, 0, A, A, None), ple.PLE_ERR_NULL),
    ((A, 2, 5, 0, A, A, A + 4), ple.PLE_ERR_ALIGN),
    ((A, 2, 5, 0, A + 2, A, A), ple.PLE_ERR_ALIGN),
    ((None, 0, 0, 0, None, None, None), ple.PLE_OK),
])
def test_validate_index_host_checks(lib, args, status):
    assert lib.ple_validate_index(*args, None) == status
