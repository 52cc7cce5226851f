"""The library's shard planner (ple_shard_plan) on the host: no GPU needed.

A batch split by token range: rank k of W takes tokens [T*k/W, T*(k+1)/W)
and the contiguous range of requests that own them (the owner of token t is
the last request whose start is at or below t, as in the token index).  The
ranges partition the tokens, and the request ranges follow from that
definition, which numpy's searchsorted restates independently."""

import numpy as np
import pytest

import layer_gram_embedding_gb300 as ple
from layer_gram_embedding_gb300 import build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def owner(cu, t):
    return int(np.searchsorted(cu.astype(np.int64), t, side="right") - 1)


def random_cu(rng, B, max_len):
    lengths = rng.integers(0, max_len + 1, size=B)
    if lengths.sum() == 0:
        lengths[0] = 1
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    return cu


@pytest.mark.parametrize("seed", range(40))
def test_plan_partitions_tokens_and_names_their_owners(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    cu = random_cu(rng, B, int(rng.choice([1, 3, 50, 1000])))
    T = int(cu[-1])
    W = int(rng.integers(1, 2 * T + 3))
    end_prev = 0
    for k in range(W):
        tb, te, rb, rc = ple.ple_shard_plan(cu, B, T, W, k)
        assert (tb, te) == (T * k // W, T * (k + 1) // W)
        assert tb == end_prev
        end_prev = te
        if te == tb:
            assert rc == 0
            continue
        assert rb == owner(cu, tb)
        assert rb + rc - 1 == owner(cu, te - 1)
        # every token of the range is owned by one of the named requests
        for t in (tb, (tb + te) // 2, te - 1):
            assert rb <= owner(cu, t) < rb + rc
    assert end_prev == T


def test_plan_of_a_decode_batch():
    for W in (1, 2, 3, 8, 9):
        spans = [ple.ple_shard_plan(None, 8, 8, W, k) for k in range(W)]
        for tb, te, rb, rc in spans:
            assert (rb, rc) == (tb, te - tb)
        assert spans[0][0] == 0 and spans[-1][1] == 8


def test_plan_rejects_bad_arguments():
    import ctypes
    cu = np.array([0, 3, 5], dtype=np.int32)
    out = [ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()]
    st = ple.lib().ple_shard_plan(cu.ctypes.data, 0, 5, 1, 0, *[ctypes.byref(o) for o in out])
    assert st == ple.PLE_ERR_SIZE  # no requests
    for args in [(cu, 2, 5, 0, 0), (cu, 2, 5, 2, 2), (cu, 2, 5, 2, -1),
                 (np.array([0, 3, 4], dtype=np.int32), 2, 5, 1, 0),   # last != T
                 (np.array([1, 3, 5], dtype=np.int32), 2, 5, 1, 0),   # first != 0
                 (np.array([0, 4, 3, 5], dtype=np.int32), 3, 5, 1, 0),  # decreasing
                 (None, 4, 5, 1, 0)]:                                  # decode needs B == T
        with pytest.raises(ple.PleError) as e:
            ple.ple_shard_plan(*args)
        assert e.value.status == ple.PLE_ERR_SIZE
    st = ple.lib().ple_shard_plan(None, 1, 1, 1, 0, None, None, None, None)
    assert st == ple.PLE_ERR_NULL


def test_shard_inputs_host_checks_before_any_launch():
    # fake, never dereferenced device addresses: each call fails a host check
    A = 0x10000
    f = ple.lib().ple_shard_inputs
    ok = dict(ids=A, dt=1, cu=A, ctx=A, B=4, T=100, C=3, tb=10, te=50, rb=0, rc=2, scu=A, sctx=A)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(a["ids"], a["dt"], a["cu"], a["ctx"], a["B"], a["T"], a["C"], a["tb"], a["te"],
                 a["rb"], a["rc"], a["scu"], a["sctx"], None)

    assert call(rb=3, rc=2) == ple.PLE_ERR_SIZE       # past the last request
    assert call(rc=0) == ple.PLE_ERR_SIZE
    assert call(te=10) == ple.PLE_ERR_SIZE            # empty range
    assert call(te=101) == ple.PLE_ERR_SIZE
    assert call(C=0) == ple.PLE_ERR_SIZE
    assert call(C=16) == ple.PLE_ERR_SIZE
    assert call(ctx=None) == ple.PLE_ERR_NULL
    assert call(dt=2) == ple.PLE_ERR_DTYPE
    assert call(sctx=A + 4) == ple.PLE_ERR_ALIGN
    assert call(scu=A + 2) == ple.PLE_ERR_ALIGN
