"""Host-only checks of the C ABI: the library builds and loads, exports every
symbol include/dsa.h declares, sizes its scratch as the pages' arithmetic
says, and rejects bad arguments before anything is enqueued (no GPU needed:
every call here fails validation, so no kernel is launched)."""
import ctypes
import os
import re

import pytest

import deepseek_v4_sparse_ratio_gb300 as dsa
from deepseek_v4_sparse_ratio_gb300 import _binding as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "dsa.h")
FAKE = 1 << 20          # an aligned non-null address; never dereferenced on the host


@pytest.fixture(scope="module")
def lib():
    dsa.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(B.EXPORTS) <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_strerror_covers_codes(lib):
    for code in range(0, -11, -1):
        assert dsa.dsa_strerror(code) != "unknown status"


def test_scratch_bytes_match_tiled_score_buffer(lib):
    # 4096 rows x 262,144 pooled rows x 4 B = 4 GiB untiled; 1 GiB for 1024-row tiles
    assert dsa.dsa_score_scratch_bytes(4096, 262144) == 4 * 2 ** 30
    assert dsa.dsa_score_scratch_bytes(1024, 262144) == 2 ** 30
    assert dsa.dsa_score_scratch_bytes(10, 129) == 10 * 256 * 4   # rows padded to 128
    assert dsa.dsa_score_scratch_bytes(0, 5) == 0


def _state(cap=100, n_pooled=0, n_tokens=0, n_rem=0, ratio=4, n_ik=None):
    return B.dsa_pool_state(FAKE, FAKE, FAKE, FAKE, cap, n_pooled,
                            n_pooled if n_ik is None else n_ik, n_tokens, n_rem, ratio)


def _append(lib, st, chunk=8, offset=0, ratio=4, raw=FAKE):
    return lib.dsa_pool_append(ctypes.byref(st), raw, raw, chunk, offset, ratio, None)


def test_pool_append_rejects_before_launch(lib):
    assert lib.dsa_pool_append(None, FAKE, FAKE, 4, 0, 4, None) == B.DSA_ERR_ARG
    st = _state()
    assert _append(lib, st, raw=None) == B.DSA_ERR_ARG
    assert _append(lib, st, chunk=0) == B.DSA_ERR_ARG
    assert _append(lib, st, raw=FAKE + 8) == B.DSA_ERR_ARG          # misaligned
    assert _append(lib, st, ratio=8) == B.DSA_ERR_SHAPE
    assert _append(lib, st, offset=4) == B.DSA_ERR_OFFSET
    st = _state(cap=10)
    assert _append(lib, st, chunk=44) == B.DSA_ERR_CAPACITY
    st = _state(n_pooled=2, n_tokens=9, n_rem=1, n_ik=3)
    assert _append(lib, st, offset=9) == B.DSA_ERR_DIVERGED
    st = _state(n_pooled=2, n_tokens=10, n_rem=1)                   # inconsistent counters
    assert _append(lib, st, offset=10) == B.DSA_ERR_ARG
    # state untouched by every failed call
    assert (st.n_pooled_kv, st.n_tokens, st.n_rem) == (2, 10, 1)


def test_score_topk_rejects_before_launch(lib):
    f = lib.dsa_index_score_topk
    # n must equal floor((offset+chunk)/4)
    assert f(FAKE, FAKE, FAKE, 5, 16, 0, 4, 2, 16, FAKE, 1 << 20, FAKE, None, None) == B.DSA_ERR_ARG
    assert f(FAKE, FAKE, FAKE, 4, 16, 0, 3, 2, 16, FAKE, 1 << 20, FAKE, None, None) == B.DSA_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, 4, 16, 0, 4, 0, 16, FAKE, 1 << 20, FAKE, None, None) == B.DSA_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, 4, 16, 0, 4, 2, 0, FAKE, 1 << 20, FAKE, None, None) == B.DSA_ERR_SHAPE
    need = dsa.dsa_score_scratch_bytes(16, 4)
    assert f(FAKE, FAKE, FAKE, 4, 16, 0, 4, 2, 16, FAKE, need - 4, FAKE, None, None) == B.DSA_ERR_SCRATCH
    assert f(FAKE, FAKE, FAKE, 4, 16, 0, 4, 2, 16, None, need, FAKE, None, None) == B.DSA_ERR_SCRATCH
    assert f(None, FAKE, FAKE, 4, 16, 0, 4, 2, 16, FAKE, need, FAKE, None, None) == B.DSA_ERR_ARG
    assert f(FAKE, FAKE, FAKE, 4, 16, 0, 4, 2, 16, FAKE, need, None, None, None) == B.DSA_ERR_ARG


def test_attention_rejects_before_launch(lib):
    f = lib.dsa_window_sparse_attn
    # raw rows must cover max(0, off-W+1) .. off+T-1
    assert f(FAKE, FAKE, 100, 200, FAKE, 50, FAKE, 8, 32, 200, 4, 128, 0.1, FAKE, None,
             None) == B.DSA_ERR_RAW_RANGE
    assert f(FAKE, FAKE, 73, 158, FAKE, 50, FAKE, 8, 32, 200, 4, 128, 0.1, FAKE, None,
             None) == B.DSA_ERR_RAW_RANGE                              # ends at 230 < 232
    assert f(FAKE, FAKE, 73, 159, FAKE, 58, FAKE, 8, 32, 200, 4, 0, 0.1, FAKE, None,
             None) == B.DSA_ERR_SHAPE
    assert f(FAKE, FAKE, 73, 159, FAKE, 58, FAKE, 8, 32, 200, 4, 128, -1.0, FAKE, None,
             None) == B.DSA_ERR_SHAPE
    assert f(FAKE, FAKE, 73, 159, FAKE, 58, None, 8, 32, 200, 4, 128, 0.1, FAKE, None,
             None) == B.DSA_ERR_ARG


def test_prefill_chunk_validates_everything_first(lib):
    st = _state(cap=1000, n_pooled=50, n_tokens=200, n_rem=0)
    f = lib.dsa_prefill_chunk
    need = dsa.dsa_score_scratch_bytes(32, 58)
    args = lambda **kw: [ctypes.byref(st), FAKE, kw.get("raw_start", 73), kw.get("raw_rows", 159),
                         FAKE, FAKE, FAKE, FAKE, 32, kw.get("offset", 200), kw.get("k", 8),
                         kw.get("window", 128), 0.1, 32, FAKE, kw.get("scratch", need), FAKE,
                         FAKE, None, None]
    assert f(*args(offset=196)) == B.DSA_ERR_OFFSET
    assert f(*args(scratch=need - 1)) == B.DSA_ERR_SCRATCH
    assert f(*args(raw_start=74)) == B.DSA_ERR_RAW_RANGE
    assert f(*args(window=0)) == B.DSA_ERR_SHAPE
    assert (st.n_pooled_kv, st.n_tokens, st.n_rem) == (50, 200, 0)


def test_wait_selftest_rejects_null_status(lib):
    assert lib.dsa_bounded_wait_selftest(0, None, None) == B.DSA_ERR_ARG


def test_host_prefill_rejects_before_any_copy(lib):
    ws = B.dsa_prefill_workspace(FAKE, 200, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20,
                                 100, 64)
    st = B.dsa_pool_state(FAKE, FAKE, FAKE, FAKE, 1000, 0, 0, 0, 0, 4)
    args = [FAKE, 0, 100, FAKE, FAKE, FAKE, FAKE, 100, 0, 64, 128, 0.05, 100, FAKE, FAKE, None,
            None, None]
    assert lib.dsa_prefill_chunk_host(ctypes.byref(st), None, *args) == B.DSA_ERR_ARG
    bad = list(args)
    bad[3] = None   # raw_ik_h
    assert lib.dsa_prefill_chunk_host(ctypes.byref(st), ctypes.byref(ws), *bad) == B.DSA_ERR_ARG
    big = list(args)
    big[7] = 101    # chunk beyond the workspace
    assert lib.dsa_prefill_chunk_host(ctypes.byref(st), ctypes.byref(ws), *big) == \
        B.DSA_ERR_CAPACITY
    big = list(args)
    big[9] = 65     # index_topk beyond the workspace
    assert lib.dsa_prefill_chunk_host(ctypes.byref(st), ctypes.byref(ws), *big) == \
        B.DSA_ERR_CAPACITY
    off = list(args)
    off[8] = 4      # offset != tokens in the cache
    assert lib.dsa_prefill_chunk_host(ctypes.byref(st), ctypes.byref(ws), *off) == \
        B.DSA_ERR_OFFSET
