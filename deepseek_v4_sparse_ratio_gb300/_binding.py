"""ctypes binding of libdsa.so: same names and argument order as include/dsa.h.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. Tensors are torch CUDA tensors (their data pointers are passed);
``stream`` defaults to torch's current stream. A non-zero return code raises
DsaError. If libdsa.so cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import buildlib as _build

RATIO, INDEX_HEADS, INDEX_DIM, HEADS, DIM = 4, 64, 128, 64, 512

DSA_OK = 0
DSA_ERR_ARG, DSA_ERR_SHAPE, DSA_ERR_OFFSET, DSA_ERR_CAPACITY = -1, -2, -3, -4
DSA_ERR_DIVERGED, DSA_ERR_SCRATCH, DSA_ERR_CUDA, DSA_ERR_TIMEOUT = -5, -6, -7, -8
DSA_ERR_BOUNDS, DSA_ERR_RAW_RANGE = -9, -10

EXPORTS = ("dsa_pool_append", "dsa_score_scratch_bytes", "dsa_index_score_topk",
           "dsa_window_sparse_attn", "dsa_prefill_chunk", "dsa_strerror",
           "dsa_index_score_topk_noalloc", "dsa_bounded_wait_selftest", "dsa_prefill_chunk_host")
DSA_STATIC_SCRATCH_BYTES = 16 << 20


class DsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {dsa_strerror(code)} (code {code})")


class dsa_pool_state(ctypes.Structure):
    _fields_ = [("pooled_kv", ctypes.c_void_p), ("pooled_ik", ctypes.c_void_p),
                ("rem_kv", ctypes.c_void_p), ("rem_ik", ctypes.c_void_p),
                ("cap", ctypes.c_int64), ("n_pooled_kv", ctypes.c_int64),
                ("n_pooled_ik", ctypes.c_int64), ("n_tokens", ctypes.c_int64),
                ("n_rem", ctypes.c_int32), ("ratio", ctypes.c_int32)]


class dsa_prefill_workspace(ctypes.Structure):
    _fields_ = [("raw_kv", ctypes.c_void_p), ("raw_kv_rows", ctypes.c_int64),
                ("raw_ik", ctypes.c_void_p), ("q_idx", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("q", ctypes.c_void_p), ("sel", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("scratch", ctypes.c_void_p), ("scratch_bytes", ctypes.c_size_t),
                ("max_chunk", ctypes.c_int64), ("max_topk", ctypes.c_int32)]


_lib = None


def load(path: str | None = None):
    """Load libdsa.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.build()
    lib = ctypes.CDLL(path)
    P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    S = ctypes.POINTER(dsa_pool_state)
    lib.dsa_pool_append.argtypes = [S, P, P, i64, i64, i32, P]
    lib.dsa_score_scratch_bytes.argtypes = [i64, i64]
    lib.dsa_score_scratch_bytes.restype = sz
    lib.dsa_index_score_topk.argtypes = [P, P, P, i64, i64, i64, i32, i32, i64, P, sz, P, P, P]
    lib.dsa_window_sparse_attn.argtypes = [P, P, i64, i64, P, i64, P, i32, i64, i64, i32, i32,
                                           ctypes.c_float, P, P, P]
    lib.dsa_prefill_chunk.argtypes = [S, P, i64, i64, P, P, P, P, i64, i64, i32, i32,
                                      ctypes.c_float, i64, P, sz, P, P, P, P]
    lib.dsa_index_score_topk_noalloc.argtypes = [P, P, P, i64, i64, i64, i32, i32, i64, P, P, P]
    lib.dsa_bounded_wait_selftest.argtypes = [i32, P, P]
    lib.dsa_prefill_chunk_host.argtypes = [S, ctypes.POINTER(dsa_prefill_workspace), P, i64, i64,
                                           P, P, P, P, i64, i64, i32, i32, ctypes.c_float, i64,
                                           P, P, P, P, P]
    lib.dsa_strerror.argtypes = [ctypes.c_int]
    lib.dsa_strerror.restype = ctypes.c_char_p
    for f in ("dsa_pool_append", "dsa_index_score_topk", "dsa_window_sparse_attn",
              "dsa_prefill_chunk", "dsa_index_score_topk_noalloc", "dsa_bounded_wait_selftest",
              "dsa_prefill_chunk_host"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != DSA_OK:
        raise DsaError(rc, where)


def dsa_strerror(code: int) -> str:
    return load().dsa_strerror(int(code)).decode()


class PoolState:
    """Caller-side PoolingCache: device buffers (torch) plus the C struct."""

    def __init__(self, cap: int, device="cuda", ratio: int = RATIO):
        self.ratio = ratio
        self.pooled_kv = torch.zeros(max(cap, 1), DIM, dtype=torch.bfloat16, device=device)
        self.pooled_ik = torch.zeros(max(cap, 1), INDEX_DIM, dtype=torch.bfloat16, device=device)
        self.rem_kv = torch.zeros(max(ratio - 1, 1), DIM, dtype=torch.bfloat16, device=device)
        self.rem_ik = torch.zeros(max(ratio - 1, 1), INDEX_DIM, dtype=torch.bfloat16, device=device)
        self.c = dsa_pool_state(self.pooled_kv.data_ptr(), self.pooled_ik.data_ptr(),
                                self.rem_kv.data_ptr(), self.rem_ik.data_ptr(), cap, 0, 0, 0, 0,
                                ratio)

    @classmethod
    def from_prefix(cls, pooled_ik, pooled_kv, n_tokens: int, cap: int, device="cuda",
                    ratio: int = RATIO):
        """A cache that already holds `pooled_*` rows after n_tokens tokens (no remainder)."""
        s = cls(cap, device, ratio)
        P = pooled_ik.shape[0]
        assert n_tokens == P * ratio and pooled_kv.shape[0] == P and P <= cap
        s.pooled_ik[:P].copy_(pooled_ik)
        s.pooled_kv[:P].copy_(pooled_kv)
        s.c.n_pooled_kv = s.c.n_pooled_ik = P
        s.c.n_tokens = n_tokens
        return s

    @property
    def n_pooled(self) -> int:
        return self.c.n_pooled_kv

    @property
    def n_tokens(self) -> int:
        return self.c.n_tokens

    @property
    def n_rem(self) -> int:
        return self.c.n_rem

    def snapshot(self):
        """O(1) rollback point: the counters and the (at most 3) remainder rows."""
        return (self.c.n_pooled_kv, self.c.n_pooled_ik, self.c.n_tokens, self.c.n_rem,
                self.rem_kv.clone(), self.rem_ik.clone())

    def restore(self, snap) -> None:
        (self.c.n_pooled_kv, self.c.n_pooled_ik, self.c.n_tokens, self.c.n_rem, rk, ri) = snap
        self.rem_kv.copy_(rk)
        self.rem_ik.copy_(ri)


def dsa_pool_append(state: PoolState, raw_kv, raw_ik, chunk: int, offset: int,
                    ratio: int | None = None, stream=None) -> None:
    ratio = state.ratio if ratio is None else ratio
    rc = load().dsa_pool_append(ctypes.byref(state.c), _p(raw_kv), _p(raw_ik), chunk, offset,
                                ratio, _s(stream))
    _check(rc, "dsa_pool_append")


def dsa_score_scratch_bytes(tile_rows: int, n_pooled: int) -> int:
    return int(load().dsa_score_scratch_bytes(tile_rows, n_pooled))


def _nbytes(t):
    if t is None:
        return 0
    return t.numel() * t.element_size()


def dsa_index_score_topk(q_idx, w, pooled_ik, n_pooled: int, chunk: int, offset: int,
                         ratio: int, index_topk: int, tile_rows: int, scratch, sel,
                         dev_status=None, stream=None) -> None:
    rc = load().dsa_index_score_topk(_p(q_idx), _p(w), _p(pooled_ik), n_pooled, chunk, offset,
                                     ratio, index_topk, tile_rows, _p(scratch), _nbytes(scratch),
                                     _p(sel), _p(dev_status), _s(stream))
    _check(rc, "dsa_index_score_topk")


def dsa_index_score_topk_noalloc(q_idx, w, pooled_ik, n_pooled: int, chunk: int, offset: int,
                                 ratio: int, index_topk: int, tile_rows: int, sel,
                                 dev_status=None, stream=None) -> None:
    """dsa_index_score_topk with the library's own score scratch (no allocation)."""
    rc = load().dsa_index_score_topk_noalloc(_p(q_idx), _p(w), _p(pooled_ik), n_pooled, chunk,
                                             offset, ratio, index_topk, tile_rows, _p(sel),
                                             _p(dev_status), _s(stream))
    _check(rc, "dsa_index_score_topk_noalloc")


def dsa_bounded_wait_selftest(arrive: bool, dev_status, stream=None) -> None:
    """Run the library's bounded mbarrier wait on a barrier that gets its arrival or none."""
    rc = load().dsa_bounded_wait_selftest(1 if arrive else 0, _p(dev_status), _s(stream))
    _check(rc, "dsa_bounded_wait_selftest")


def dsa_window_sparse_attn(q, raw_kv, raw_start: int, pooled_kv, n_pooled: int, sel,
                           index_topk: int, chunk: int, offset: int, ratio: int, window: int,
                           scale: float, out, dev_status=None, stream=None,
                           raw_rows: int | None = None) -> None:
    rows = raw_kv.shape[0] if raw_rows is None else raw_rows
    rc = load().dsa_window_sparse_attn(_p(q), _p(raw_kv), raw_start, rows, _p(pooled_kv),
                                       n_pooled, _p(sel), index_topk, chunk, offset, ratio,
                                       window, scale, _p(out), _p(dev_status), _s(stream))
    _check(rc, "dsa_window_sparse_attn")


def dsa_prefill_chunk(state: PoolState, raw_kv, raw_start: int, raw_ik, q_idx, w, q,
                      chunk: int, offset: int, index_topk: int, window: int, scale: float,
                      tile_rows: int, scratch, sel, out, dev_status=None, stream=None,
                      raw_rows: int | None = None) -> None:
    rows = raw_kv.shape[0] if raw_rows is None else raw_rows
    rc = load().dsa_prefill_chunk(ctypes.byref(state.c), _p(raw_kv), raw_start, rows,
                                  _p(raw_ik), _p(q_idx), _p(w), _p(q), chunk, offset, index_topk,
                                  window, scale, tile_rows, _p(scratch), _nbytes(scratch),
                                  _p(sel), _p(out), _p(dev_status), _s(stream))
    _check(rc, "dsa_prefill_chunk")


class PrefillWorkspace:
    """Device buffers for dsa_prefill_chunk_host (torch allocations, caller-owned)."""

    def __init__(self, max_chunk: int, max_topk: int, raw_kv_rows: int, n_pooled_max: int,
                 tile_rows: int, device="cuda"):
        dev = torch.device(device)
        self.raw_kv = torch.empty(raw_kv_rows, DIM, dtype=torch.bfloat16, device=dev)
        self.raw_ik = torch.empty(max_chunk, INDEX_DIM, dtype=torch.bfloat16, device=dev)
        self.q_idx = torch.empty(max_chunk, INDEX_HEADS, INDEX_DIM, dtype=torch.bfloat16,
                                 device=dev)
        self.w = torch.empty(max_chunk, INDEX_HEADS, dtype=torch.float32, device=dev)
        self.q = torch.empty(max_chunk, HEADS, DIM, dtype=torch.bfloat16, device=dev)
        self.sel = torch.empty(max_chunk, max_topk, dtype=torch.int32, device=dev)
        self.out = torch.empty(max_chunk, HEADS, DIM, dtype=torch.bfloat16, device=dev)
        nbytes = dsa_score_scratch_bytes(min(tile_rows, max_chunk), n_pooled_max)
        self.scratch = torch.empty(max(nbytes // 4, 1), dtype=torch.float32, device=dev)
        self.c = dsa_prefill_workspace(
            self.raw_kv.data_ptr(), raw_kv_rows, self.raw_ik.data_ptr(), self.q_idx.data_ptr(),
            self.w.data_ptr(), self.q.data_ptr(), self.sel.data_ptr(), self.out.data_ptr(),
            self.scratch.data_ptr(), self.scratch.numel() * 4, max_chunk, max_topk)


def dsa_prefill_chunk_host(state: "PoolState", ws: PrefillWorkspace, raw_kv_h, raw_start: int,
                           raw_ik_h, q_idx_h, w_h, q_h, chunk: int, offset: int,
                           index_topk: int, window: int, scale: float, tile_rows: int,
                           sel_h, out_h, dev_status=None, stream=None,
                           copy_stream=None) -> None:
    """The whole path from host tensors (pinned for overlap) to host tensors."""
    rc = load().dsa_prefill_chunk_host(
        ctypes.byref(state.c), ctypes.byref(ws.c), _p(raw_kv_h), raw_start, raw_kv_h.shape[0],
        _p(raw_ik_h), _p(q_idx_h), _p(w_h), _p(q_h), chunk, offset, index_topk, window, scale,
        tile_rows, _p(sel_h), _p(out_h), _p(dev_status), _s(stream),
        _s(copy_stream) if copy_stream is not None else _s(stream))
    _check(rc, "dsa_prefill_chunk_host")
