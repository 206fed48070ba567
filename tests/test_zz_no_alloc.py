"""dsa_index_score_topk_noalloc: the score + top-k step for callers that cannot
allocate device memory when they call in (a plugin handed only tensor pointers,
a server with a fixed device-memory budget). It keeps its score scratch in an
array inside libdsa.so, so the caller passes only inputs and outputs.

Checked through the C ABI, call after call on the same shared array (which
keeps the previous call's contents): against the oracle (scores + top-k on
every row, tie-band rule) and against dsa_index_score_topk with a caller-owned
scratch (the same kernels, so the same selection bit for bit). The cases cover
a single tile, several tiles, a small tile after a larger one, and the skip
path (every pooled row fits index_topk, nothing is scored). A tile larger than
the array must be refused before anything runs. This file is collected last on
purpose.
"""
import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_sparse_ratio_gb300 import _binding as B

from parity import check_selection

pytestmark = pytest.mark.gpu


def _case(seed, off, T):
    g = torch.Generator().manual_seed(seed)
    n = (off + T) // 4
    q_idx = torch.randn(T, 64, 128, generator=g).to(torch.bfloat16)
    w = torch.randn(T, 64, generator=g) * 0.125
    pik = torch.randn(n, 128, generator=g).to(torch.bfloat16)
    return q_idx, w, pik, n


def _with_caller_scratch(q_idx, w, pik, n, T, off, k, tile):
    sel = torch.empty(T, k, dtype=torch.int32, device="cuda")
    nbytes = max(B.dsa_score_scratch_bytes(min(tile, T), n), 4)
    scratch = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    B.dsa_index_score_topk(q_idx, w, pik, n, T, off, 4, k, tile, scratch, sel)
    return sel


# (seed, offset, chunk, index_topk, tile_rows): one tile; several tiles; a smaller
# tile after larger ones; the skip path (n <= index_topk)
CASES = [(101, 4096, 300, 256, 300), (202, 20000, 517, 1024, 128),
         (303, 8000, 700, 256, 64), (404, 400, 300, 256, 64)]


def test_no_alloc_matches_oracle_and_caller_scratch_call_after_call(dsa):
    lib = B.load()
    for seed, off, T, k, tile in CASES:
        q_idx, w, pik, n = _case(seed, off, T)
        assert B.dsa_score_scratch_bytes(min(tile, T), n) <= B.DSA_STATIC_SCRATCH_BYTES
        dq, dw, dk = q_idx.cuda(), w.cuda(), pik.cuda()
        sel = torch.full((T, k), 7, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = lib.dsa_index_score_topk_noalloc(dq.data_ptr(), dw.data_ptr(), dk.data_ptr(), n,
                                              T, off, 4, k, tile, sel.data_ptr(),
                                              status.data_ptr(),
                                              torch.cuda.current_stream().cuda_stream)
        assert rc == 0, B.dsa_strerror(rc)
        torch.cuda.synchronize()
        assert status.item() == 0
        got = sel.cpu().numpy()
        pos = off + np.arange(T)
        ref_sel, ref_s, mag = oracle.select(q_idx, w.numpy(), pos, pik, n, 4, k)
        check_selection(got, ref_sel, pos, n, k, ref_s, mag)
        if n <= k:
            assert ref_s is None and np.array_equal(got, ref_sel)   # skip path: exact
        ref = _with_caller_scratch(dq, dw, dk, n, T, off, k, tile)
        assert torch.equal(sel, ref)


def test_no_alloc_refuses_a_tile_beyond_the_array(dsa):
    lib = B.load()
    off, T, k = 1044480, 4096, 2048
    n = (off + T) // 4
    too_big = B.dsa_score_scratch_bytes(1024, n)
    assert too_big > B.DSA_STATIC_SCRATCH_BYTES
    fake = 1 << 20   # validation fails before any pointer is used
    rc = lib.dsa_index_score_topk_noalloc(fake, fake, fake, n, T, off, 4, k, 1024, fake, None, None)
    assert rc == B.DSA_ERR_SCRATCH
