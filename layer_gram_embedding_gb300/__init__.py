"""GB300 (sm_103a) PLE n-gram row-id hash.

The compute lives in libple.so (hand-written CUDA kernels behind the C ABI of
include/ple.h); this package is its thin Python binding.  Importing it loads
nothing; the library is loaded on the first call and its absence is an error,
never a fallback.
"""

from .binding import (PLE_ERR_ALIGN, PLE_ERR_CUDA, PLE_ERR_DTYPE, PLE_ERR_GEOMETRY_CTX,
                      PLE_ERR_GEOMETRY_HEADS, PLE_ERR_NULL, PLE_ERR_SIZE, PLE_I32, PLE_I64,
                      PLE_HEAD_BYTES, PLE_MAX_EMBED_DIM, PLE_MAX_HEADS, PLE_MAX_NGRAM, PLE_OK,
                      PleError, lib, ple_build_token_index, ple_prepare_heads, ple_row_embed,
                      ple_row_ids, ple_shard_inputs, ple_shard_plan,
                      ple_selftest_floor_mod, ple_validate_index, set_programmatic_launch,
                      small_batch_max_rows, status_string)

from .index_cache import TokenIndexCache

__all__ = [
    "TokenIndexCache",
    "PLE_OK", "PLE_ERR_NULL", "PLE_ERR_SIZE", "PLE_ERR_GEOMETRY_CTX", "PLE_ERR_GEOMETRY_HEADS",
    "PLE_ERR_DTYPE", "PLE_ERR_ALIGN", "PLE_ERR_CUDA", "PLE_I32", "PLE_I64", "PLE_MAX_NGRAM",
    "PLE_MAX_HEADS", "PLE_MAX_EMBED_DIM", "PLE_HEAD_BYTES", "PleError", "lib", "status_string",
    "small_batch_max_rows", "set_programmatic_launch",
    "ple_build_token_index", "ple_prepare_heads", "ple_row_ids", "ple_row_embed",
    "ple_shard_plan", "ple_shard_inputs",
    "ple_selftest_floor_mod",
    "ple_validate_index",
]
