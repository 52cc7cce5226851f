"""GPU: the row-id hash at the largest sizes the C ABI accepts.

- T = 2^31 - 1 tokens (the largest num_tokens): the output offsets
  ((l * T + t) * H) and the tile indices pass 2^31, so every index
  computation must be 64-bit.  The ids are drawn on the device (seeded) and
  the oracle is compared on sampled windows copied back, each hashed as a
  batch of its own with the context it carries.
- L = 70000 layers in one call: more layer groups than a grid's y dimension
  (65535) could take one per block, so the layers are grouped.
- L = 65535 layers through the small-batch kernel (one layer per grid.y).

Expected values come from the oracle only."""

import numpy as np
import pytest
import torch

import layer_gram_embedding_gb300 as ple
import oracle
import workloads as wl

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = torch.device("cuda:0")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def test_largest_token_count():
    if torch.cuda.get_device_properties(DEV).total_memory < 40 * 2 ** 30:
        pytest.skip("needs about 30 GB of device memory")
    T = 2 ** 31 - 1
    N, hpn, L = 2, 1, 1  # H = 1: 8 bytes of row ids a token
    rng = np.random.default_rng(71)
    M = wl.signed_multipliers(rng, L, N)
    vocab = wl.random_primes(rng, L * hpn, 2 ** 17, 2 ** 20).reshape(L, hpn)
    off = wl.prefix_offsets(vocab) + 12345
    b = 151643
    ctx = np.array([[b]], dtype=np.int32)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(71)
    ids = torch.randint(0, 151936, (T,), dtype=torch.int32, device=DEV, generator=gen)
    # boundaries at every 97th token, so windows cross them
    ids[::97] = b
    cu = torch.tensor([0, T], dtype=torch.int32, device=DEV)
    out = torch.empty((L, T, 1), dtype=torch.int64, device=DEV)
    ple.ple_row_ids(ids, None, None, dev(ctx), dev(M), dev(vocab), dev(off), N, hpn, b, out=out,
                    cu_seqlens=cu)
    torch.cuda.synchronize()
    picks = sorted({0, 1, 96, 97, 98, T - 1, T - 2, 2 ** 31 - 64, 2 ** 30, 2 ** 30 + 1,
                    *rng.integers(0, T, size=200).tolist()})
    for t in picks:
        a = max(0, t - (N - 1))
        seg = ids[a:t + 1].cpu().numpy()
        # the window of token t needs the N - 1 ids before it: a one-request
        # batch of tokens a..t whose context is the ids before a (or the
        # request's context at the start)
        if a == 0:
            c = ctx
        else:
            c = ids[a - (N - 1):a].cpu().numpy().reshape(1, N - 1)
        req = np.zeros(seg.shape[0], dtype=np.int32)
        local = np.arange(seg.shape[0], dtype=np.int32)
        expect = oracle.row_ids(seg, req, local, c, M, vocab, off, N, hpn, b)[0, -1, 0]
        got = int(out[0, t, 0])
        assert got == expect, (t, got, expect)


@pytest.mark.parametrize("L,T,N,hpn", [(70000, 64, 3, 1), (65535, 1, 2, 1)])
def test_most_layers_in_one_call(L, T, N, hpn):
    """70000 layers take the tiled kernel with grouped layers; 65535 layers
    of a one-token call take the small-batch kernel, one layer per grid.y."""
    rng = np.random.default_rng(L)
    H = (N - 1) * hpn
    M = wl.signed_multipliers(rng, L, N)
    vocab = wl.random_primes(rng, 64, 2 ** 17, 2 ** 20)[rng.integers(0, 64, size=L * H)]
    vocab = vocab.reshape(L, H)
    off = wl.prefix_offsets(vocab)
    batch = wl.Batch(f"layers_{L}", wl.uniform_ids(rng, T, 0.1),
                     wl.uniform_ids(rng, N - 1, 0.1).reshape(1, N - 1),
                     wl.cu_from_lengths([T]), False, M, vocab, off, N, hpn)
    assert (batch.row_ids_per_call > ple.small_batch_max_rows()) == (L == 70000)
    got = ple.ple_row_ids(dev(batch.ids), None, None, dev(batch.ngram_context), dev(M),
                          dev(vocab), dev(off), N, hpn, batch.boundary_id,
                          cu_seqlens=dev(batch.cu_seqlens))
    req, local = oracle.token_index(batch.cu_seqlens, 1, T, False)
    expect = oracle.row_ids(batch.ids, req, local, batch.ngram_context, M, vocab, off, N, hpn,
                            batch.boundary_id)
    assert np.array_equal(got.cpu().numpy(), expect)
