"""DeepSeek-V4 indexed sparse attention for chunked prefill, on one GB300 (sm_103a).

The path (pool/append -> indexer score + top-k -> window + selected attention)
runs in the CUDA kernels of libdsa.so behind the C ABI in include/dsa.h; this
package holds the in-tree build step and a thin ctypes binding with the same
function names. There is no CPU fallback: calls raise if the library is missing.
"""
from .buildlib import build as _build_lib
from ._binding import (DIM, HEADS, INDEX_DIM, INDEX_HEADS, RATIO, DsaError, PoolState,  # noqa: F401
                       PrefillWorkspace, dsa_bounded_wait_selftest, dsa_index_score_topk,
                       dsa_index_score_topk_noalloc, dsa_pool_append, dsa_prefill_chunk,
                       dsa_prefill_chunk_host,
                       dsa_score_scratch_bytes, dsa_strerror, dsa_window_sparse_attn, load)


def build(force: bool = False) -> str:
    """Compile libdsa.so for sm_103a (if stale) and load it."""
    path = _build_lib(force=force)
    load(path)
    return path
