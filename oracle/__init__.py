"""CPU oracle for DeepSeek-V4 indexed sparse attention in a chunked prefill.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg call this package; the library never does. It
shares no code with the CUDA path. The arithmetic lives in ``dsa_oracle.c``
(fp64 accumulation, one rounding to the output type); this module holds the
PoolingCache state machine and array marshalling.

State machine (first page, "perf(deepseek-v4): skip redundant all-pooled
indexer scoring", Summary and Correctness): after N tokens the cache holds
floor(N/ratio) pooled rows and the last N mod ratio raw rows as a remainder;
the attention-KV and indexer-key compressors advance together, and their row
counts must agree.

Selection (same page, Summary): when 0 < n <= index_topk the scoring is
skipped and the selection is the sequential indices; the full path is kept
for empty pools and for n > index_topk.

Parity: every function here is pinned in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile dsa_oracle.c into liboracle.so with gcc (OpenMP, no FP contraction,
    no reassociation: -O3 only vectorises loops whose sums stay independent)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O3", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        lib.dsa_oracle_round_bf16.argtypes = [f64]
        lib.dsa_oracle_round_bf16.restype = ctypes.c_uint16
        lib.dsa_oracle_pool_rows.argtypes = [P, i64, i32, i32, P]
        lib.dsa_oracle_index_scores.argtypes = [P, P, P, i64, P, i64, i32, i32, i32, P, P]
        lib.dsa_oracle_topk.argtypes = [P, P, i64, i64, i32, i32, P]
        lib.dsa_oracle_attention.argtypes = [P, P, i64, P, i64, i64, P, i64, P, i32, i32,
                                             i32, i32, f64, P]
        lib.dsa_oracle_attention.restype = ctypes.c_int
        lib.dsa_oracle_round_bf16_array.argtypes = [P, i64, P]
        lib.dsa_oracle_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def as_bf16_bits(x) -> np.ndarray:
    """torch bf16 tensor (or uint16 array) -> C-contiguous uint16 bit array."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy().view(np.uint16))


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def threads() -> int:
    return int(_load().dsa_oracle_threads())


def round_bf16(x: float) -> int:
    """bf16 bit pattern of x under round-to-nearest-even."""
    return int(_load().dsa_oracle_round_bf16(float(x)))


def round_bf16_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().dsa_oracle_round_bf16_array(_ptr(x), x.size, _ptr(out))
    return out


def n_vis(t, ratio: int, n: int):
    """Pooled rows visible to absolute position t (pooled row j covers tokens
    j*ratio..j*ratio+ratio-1 and becomes visible at its last token)."""
    return np.minimum((np.asarray(t, dtype=np.int64) + 1) // ratio, n)


def pool_rows(src: np.ndarray, ratio: int) -> np.ndarray:
    """Mean-pool complete groups of `ratio` consecutive rows of src [G*ratio, dim]."""
    src = as_bf16_bits(src)
    rows, dim = src.shape
    assert rows % ratio == 0
    out = np.empty((rows // ratio, dim), dtype=np.uint16)
    if rows:
        _load().dsa_oracle_pool_rows(_ptr(src), rows // ratio, dim, ratio, _ptr(out))
    return out


class PoolState:
    """The oracle's PoolingCache: pooled rows of both streams, the raw remainder
    of both streams, and the token count."""

    def __init__(self, ratio: int = 4, dim_ik: int = 128, dim_kv: int = 512):
        self.ratio = ratio
        self.pooled_ik = np.zeros((0, dim_ik), np.uint16)
        self.pooled_kv = np.zeros((0, dim_kv), np.uint16)
        self.rem_ik = np.zeros((0, dim_ik), np.uint16)
        self.rem_kv = np.zeros((0, dim_kv), np.uint16)
        self.n_tokens = 0

    @classmethod
    def from_prefix(cls, pooled_ik, pooled_kv, n_tokens: int, ratio: int = 4):
        """A cache holding given pooled rows after n_tokens tokens (no remainder)."""
        pi, pk = as_bf16_bits(pooled_ik), as_bf16_bits(pooled_kv)
        s = cls(ratio, dim_ik=pi.shape[1], dim_kv=pk.shape[1])
        s.pooled_ik = pi.copy()
        s.pooled_kv = pk.copy()
        assert n_tokens % ratio == 0 and s.pooled_ik.shape[0] == n_tokens // ratio
        s.n_tokens = n_tokens
        return s

    @property
    def n_pooled(self) -> int:
        assert self.pooled_ik.shape[0] == self.pooled_kv.shape[0], "compressors diverged"
        return self.pooled_ik.shape[0]

    @property
    def n_rem(self) -> int:
        return self.rem_ik.shape[0]

    def copy(self) -> "PoolState":
        s = PoolState(self.ratio, self.pooled_ik.shape[1], self.pooled_kv.shape[1])
        s.pooled_ik, s.pooled_kv = self.pooled_ik.copy(), self.pooled_kv.copy()
        s.rem_ik, s.rem_kv = self.rem_ik.copy(), self.rem_kv.copy()
        s.n_tokens = self.n_tokens
        return s

    def append(self, raw_ik, raw_kv, offset: int) -> None:
        """Run both compressors over one chunk of raw rows at absolute `offset`."""
        if offset != self.n_tokens:
            raise ValueError(f"offset {offset} != tokens seen {self.n_tokens}")
        raw_ik, raw_kv = as_bf16_bits(raw_ik), as_bf16_bits(raw_kv)
        assert raw_ik.shape[0] == raw_kv.shape[0]
        r = self.ratio
        for name in ("ik", "kv"):
            rows = np.concatenate([getattr(self, "rem_" + name),
                                   raw_ik if name == "ik" else raw_kv], axis=0)
            full = (rows.shape[0] // r) * r
            new = pool_rows(rows[:full], r)
            setattr(self, "pooled_" + name,
                    np.concatenate([getattr(self, "pooled_" + name), new], axis=0))
            setattr(self, "rem_" + name, rows[full:].copy())
        self.n_tokens += raw_ik.shape[0]
        assert self.n_pooled == self.n_tokens // r and self.n_rem == self.n_tokens % r


def index_scores(q_idx, w, pos, pooled_ik, n: int, ratio: int = 4):
    """Masked indexer scores (fp32) and term magnitudes (fp64), both [R, n]."""
    q_idx = as_bf16_bits(q_idx)
    R, heads, dim = q_idx.shape
    w = np.ascontiguousarray(np.asarray(w, dtype=np.float32))
    pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int64))
    k = as_bf16_bits(pooled_ik)[:n]
    k = np.ascontiguousarray(k)
    assert w.shape == (R, heads) and pos.shape == (R,) and k.shape == (n, dim)
    scores = np.empty((R, n), np.float32)
    mag = np.empty((R, n), np.float64)
    if R and n:
        _load().dsa_oracle_index_scores(_ptr(q_idx), _ptr(w), _ptr(pos), R, _ptr(k), n,
                                        heads, dim, ratio, _ptr(scores), _ptr(mag))
    return scores, mag


def topk(scores: np.ndarray, pos, n: int, ratio: int, k: int) -> np.ndarray:
    """Ascending, -1 padded top-k indices [R, k] under (score desc, index asc)."""
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int64))
    R = pos.shape[0]
    assert scores.shape == (R, n)
    sel = np.empty((R, k), np.int32)
    if R:
        _load().dsa_oracle_topk(_ptr(scores), _ptr(pos), R, n, ratio, k, _ptr(sel))
    return sel


def sequential_selection(pos, n: int, ratio: int, k: int) -> np.ndarray:
    """Selection of the all-pooled skip path: 0..n_vis-1, -1 padded."""
    nv = n_vis(pos, ratio, n)
    ar = np.arange(k, dtype=np.int64)[None, :]
    return np.where(ar < nv[:, None], ar, -1).astype(np.int32)


def select(q_idx, w, pos, pooled_ik, n: int, ratio: int, k: int, force_full: bool = False):
    """Selection for rows at `pos` after the append: skip path when 0 < n <= k
    (unless force_full), else score + top-k. Returns (sel, scores, mag) with
    scores/mag None on the skip path."""
    R = len(pos)
    if n == 0:
        return np.full((R, k), -1, np.int32), None, None
    if n <= k and not force_full:
        return sequential_selection(pos, n, ratio, k), None, None
    s, m = index_scores(q_idx, w, pos, pooled_ik, n, ratio)
    return topk(s, pos, n, ratio, k), s, m


def attention(q, pos, raw_kv, raw_start: int, pooled_kv, n: int, sel, window: int,
              scale: float) -> np.ndarray:
    """fp64 window + selected-pooled attention [R, H, D]."""
    q = as_bf16_bits(q)
    R, heads, dim = q.shape
    pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int64))
    raw = as_bf16_bits(raw_kv)
    pk = np.ascontiguousarray(as_bf16_bits(pooled_kv)[:max(n, 0)])
    if pk.shape[0] == 0:
        pk = np.zeros((1, dim), np.uint16)
    sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int32))
    k = sel.shape[1]
    out = np.empty((R, heads, dim), np.float64)
    if R:
        rc = _load().dsa_oracle_attention(_ptr(q), _ptr(pos), R, _ptr(raw), raw_start,
                                          raw.shape[0], _ptr(pk), n, _ptr(sel), k, window,
                                          heads, dim, float(scale), _ptr(out))
        if rc != 0:
            raise ValueError("attention: a key row lies outside the given buffers")
    return out


def prefill_chunk(state: PoolState, raw_ik, raw_kv_chunk, offset: int, q_idx, w, q,
                  raw_kv_all, raw_start: int, rows, k: int, window: int, scale: float,
                  force_full: bool = False, want_attention: bool = True):
    """One chunk of the whole path for the chunk-local rows `rows`:
    append (both compressors), select, attend. Returns a dict."""
    state.append(raw_ik, raw_kv_chunk, offset)
    n = state.n_pooled
    rows = np.asarray(rows, dtype=np.int64)
    pos = offset + rows
    qi = as_bf16_bits(q_idx)[rows]
    ww = np.asarray(w, dtype=np.float32)[rows]
    sel, scores, mag = select(qi, ww, pos, state.pooled_ik, n, state.ratio, k, force_full)
    res = {"n": n, "sel": sel, "scores": scores, "mag": mag, "pos": pos}
    if want_attention:
        res["out"] = attention(as_bf16_bits(q)[rows], pos, raw_kv_all, raw_start,
                               state.pooled_kv, n, sel, window, scale)
    return res
