"""The token-index memo (host logic): the page's memo tests, on CPU with a
counting fake builder, plus a GPU check with the library's builder.

FreeToken PR #338 ("perf(ple): fuse the n-gram row-id hash into one Triton
kernel", sections "Why it is safe" and "How it was tested"): the index is
memoized per (is_decode, shape, device), bounded, not cached while a CUDA
graph is captured, and a decode is never confused with a one-request prefill.
"""

import numpy as np
import pytest
import torch

from layer_gram_embedding_gb300 import index_cache
from layer_gram_embedding_gb300.index_cache import TokenIndexCache


class FakeBuilder:
    def __init__(self):
        self.calls = []

    def __call__(self, lengths, is_decode, device):
        self.calls.append((lengths, is_decode, str(device)))
        return ("req", lengths, is_decode), ("local", len(self.calls))


def test_cache_is_keyed_by_shape():
    f = FakeBuilder()
    c = TokenIndexCache(builder=f)
    a = c.get([3, 5], False, "cpu")
    assert c.get([3, 5], False, "cpu") is a
    b = c.get([5, 3], False, "cpu")
    assert b is not a and len(f.calls) == 2
    assert c.get([3, 5], False, "cuda:0") is not a  # the device is part of the key
    assert (c.hits, c.misses) == (1, 3)


def test_cache_is_bounded_lru():
    f = FakeBuilder()
    c = TokenIndexCache(capacity=3, builder=f)
    for n in range(1, 6):
        c.get([n], False, "cpu")
    assert len(c) == 3
    c.get([3], False, "cpu")           # still cached: a hit
    assert len(f.calls) == 5
    c.get([1], False, "cpu")           # evicted: rebuilt
    assert len(f.calls) == 6 and len(c) == 3


def test_decode_is_not_confused_with_a_one_request_prefill():
    f = FakeBuilder()
    c = TokenIndexCache(builder=f)
    dec = c.get([1, 1, 1, 1], True, "cpu")
    pre = c.get([4], False, "cpu")
    one_token_prefills = c.get([1, 1, 1, 1], False, "cpu")
    assert len({id(dec), id(pre), id(one_token_prefills)}) == 3
    assert [x[1] for x in f.calls] == [True, False, False]
    with pytest.raises(ValueError):
        c.get([2, 1], True, "cpu")


def test_builds_during_capture_are_not_cached(monkeypatch):
    f = FakeBuilder()
    c = TokenIndexCache(builder=f)
    monkeypatch.setattr(index_cache, "_capturing", lambda: True)
    c.get([7], False, "cpu")
    c.get([7], False, "cpu")
    assert len(f.calls) == 2 and len(c) == 0
    monkeypatch.setattr(index_cache, "_capturing", lambda: False)
    c.get([7], False, "cpu")
    assert len(c) == 1


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_cache_with_the_library_builder():
    import oracle
    import workloads as wl

    dev = torch.device("cuda:0")
    c = TokenIndexCache()
    batch = wl.ragged_16()
    lengths = np.diff(batch.cu_seqlens).tolist()
    req, local = c.get(lengths, False, dev)
    oreq, olocal = oracle.token_index(batch.cu_seqlens, batch.num_requests, batch.num_tokens,
                                      False)
    assert np.array_equal(req.cpu().numpy(), oreq) and np.array_equal(local.cpu().numpy(), olocal)
    again = c.get(lengths, False, dev)
    assert again[0].data_ptr() == req.data_ptr()  # a replay reads a stable address
    dreq, dlocal = c.get([1] * 8, True, dev)
    assert dreq.cpu().tolist() == list(range(8)) and dlocal.cpu().tolist() == [0] * 8
