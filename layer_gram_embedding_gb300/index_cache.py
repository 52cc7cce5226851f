"""Memo of per-batch-shape token indexes (host logic only).

FreeToken PR #338 ("perf(ple): fuse the n-gram row-id hash into one Triton
kernel", section "Why it is safe") memoizes the (request, offset) index the
fused kernel addresses through: keyed by (is_decode, shape, device), so that
a CUDA-graph replay reads a stable address; a build that happens during
graph capture is not cached (its buffers live in the graph's pool); the memo
is bounded.  is_decode is part of the key because a decode of B requests and
a prefill of one B-token request have the same [T] and opposite meanings.

Here the batch shape is the tuple of request lengths (a decode's is B ones,
which the flag keeps apart from a one-request prefill of B tokens).  The
index itself is always built by the library's ple_build_token_index; this
class only decides when to reuse one.
"""

from __future__ import annotations

from collections import OrderedDict
from typing import Callable, Sequence

import torch

DEFAULT_CAPACITY = 64


def _capturing() -> bool:
    return torch.cuda.is_available() and torch.cuda.is_current_stream_capturing()


class TokenIndexCache:
    """Bounded LRU memo of (req, local) device tensors per batch shape.

    `builder(cu_seqlens, num_requests, num_tokens, is_decode, device)` makes a
    fresh index; the default is the library's ple_build_token_index.
    """

    def __init__(self, capacity: int = DEFAULT_CAPACITY, builder: Callable | None = None):
        if capacity < 1:
            raise ValueError("capacity must be at least 1")
        self.capacity = int(capacity)
        self._builder = builder
        self._entries: OrderedDict = OrderedDict()
        self.hits = 0
        self.misses = 0

    def __len__(self) -> int:
        return len(self._entries)

    def _build(self, lengths, is_decode, device, cu_seqlens):
        if self._builder is not None:
            return self._builder(lengths, is_decode, device)
        from .binding import ple_build_token_index

        T = int(sum(lengths))
        B = len(lengths)
        cu = None
        if not is_decode:
            if cu_seqlens is not None:
                cu = cu_seqlens
            elif _capturing():
                raise RuntimeError("a prefill index built during CUDA-graph capture needs its "
                                   "cu_seqlens on the device; build it once before capture")
            else:
                cu_host = torch.zeros(B + 1, dtype=torch.int32)
                cu_host[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(
                    torch.int32)
                cu = cu_host.to(device)
        return ple_build_token_index(cu, B, T, is_decode, device=device)

    def get(self, lengths: Sequence[int], is_decode: bool, device,
            cu_seqlens: torch.Tensor | None = None) -> tuple:
        """(req, local) for a batch whose request lengths are `lengths` (host
        integers; a decode passes B ones).  Reused when the same shape was
        seen on the same device; never stored while a CUDA graph is being
        captured.  `cu_seqlens` (the lengths' prefix sums, int32 on the
        device) saves an upload on a miss and is required for a prefill
        miss during capture."""
        lengths = tuple(int(x) for x in lengths)
        if is_decode and any(x != 1 for x in lengths):
            raise ValueError("a decode has exactly one token per request")
        device = torch.device(device)
        key = (bool(is_decode), lengths, str(device))
        hit = self._entries.get(key)
        if hit is not None:
            self._entries.move_to_end(key)
            self.hits += 1
            return hit
        self.misses += 1
        index = self._build(lengths, bool(is_decode), device, cu_seqlens)
        if not _capturing():
            self._entries[key] = index
            while len(self._entries) > self.capacity:
                self._entries.popitem(last=False)
        return index

    def clear(self) -> None:
        self._entries.clear()
