"""dsa_index_score_topk_noalloc: the score + top-k step for callers that cannot
allocate device memory when they call in (a plugin handed only tensor pointers,
a server with a fixed device-memory budget). It keeps its score scratch in an
array inside libdsa.so, so the caller passes only inputs and outputs.

Checked through the C ABI against dsa_index_score_topk with a caller-owned
scratch: two calls in a row on different inputs (the shared array keeps the
previous call's contents) must give the same selection, and a tile larger
than the array must be refused before anything runs. This file is collected
last on purpose.
"""
import ctypes

import pytest
import torch

from deepseek_v4_sparse_ratio_gb300 import _binding as B

pytestmark = pytest.mark.gpu


def _case(seed, off, T):
    g = torch.Generator().manual_seed(seed)
    n = (off + T) // 4
    q_idx = torch.randn(T, 64, 128, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(T, 64, generator=g) * 0.125).cuda()
    pik = torch.randn(n, 128, generator=g).to(torch.bfloat16).cuda()
    return q_idx, w, pik, n


def _with_caller_scratch(q_idx, w, pik, n, T, off, k, tile):
    sel = torch.empty(T, k, dtype=torch.int32, device="cuda")
    scratch = torch.empty(B.dsa_score_scratch_bytes(min(tile, T), n) // 4, dtype=torch.float32,
                          device="cuda")
    B.dsa_index_score_topk(q_idx, w, pik, n, T, off, 4, k, tile, scratch, sel)
    return sel


def test_no_alloc_matches_caller_scratch_twice(dsa):
    lib = B.load()
    cases = [(101, 4096, 300, 256, 300), (202, 20000, 517, 1024, 128)]
    for seed, off, T, k, tile in cases:
        q_idx, w, pik, n = _case(seed, off, T)
        assert B.dsa_score_scratch_bytes(min(tile, T), n) <= B.DSA_STATIC_SCRATCH_BYTES
        ref = _with_caller_scratch(q_idx, w, pik, n, T, off, k, tile)
        sel = torch.full((T, k), 7, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = lib.dsa_index_score_topk_noalloc(q_idx.data_ptr(), w.data_ptr(), pik.data_ptr(), n,
                                              T, off, 4, k, tile, sel.data_ptr(),
                                              status.data_ptr(),
                                              torch.cuda.current_stream().cuda_stream)
        assert rc == 0, B.dsa_strerror(rc)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert torch.equal(sel, ref)   # the selection is exact (and tile-independent)


def test_no_alloc_refuses_a_tile_beyond_the_array(dsa):
    lib = B.load()
    off, T, k = 1044480, 4096, 2048
    n = (off + T) // 4
    too_big = B.dsa_score_scratch_bytes(1024, n)
    assert too_big > B.DSA_STATIC_SCRATCH_BYTES
    fake = 1 << 20   # validation fails before any pointer is used
    rc = lib.dsa_index_score_topk_noalloc(fake, fake, fake, n, T, off, 4, k, 1024, fake, None, None)
    assert rc == B.DSA_ERR_SCRATCH
