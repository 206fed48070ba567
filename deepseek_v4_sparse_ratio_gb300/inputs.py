"""Seeded synthetic workloads for the indexed sparse prefill path.

This module draws random inputs and nothing else: it holds none of the
method's arithmetic (no pooling, scoring, selection or attention), so both the
CPU oracle and the CUDA path can take their inputs from it.

Shapes and distributions follow the workloads the pages discuss for
DeepSeek-V4 chunked prefill ("perf(deepseek-v4): skip redundant all-pooled
indexer scoring", Performance evidence: 2,048-token prefill steps; "[Discussion]
Tile indexed-attention scoring independently of the global prefill chunk",
128 GB / 1M-context motivation: a 4,096-token global chunk at 1,048,576 tokens
of context): B=1, indexer heads H_I=64 of dim
d_I=128, attention heads H=64 over one shared KV row of dim D=512, all values
drawn ~N(0,1) in fp32 and rounded to bf16, indexer head weights ~N(0,1/64) kept
in fp32.

Draw order (fixed, so that chunking never changes an input): raw_ik [L,128],
raw_kv [L,512], q_idx [L,64,128], w [L,64], q [L,64,512]; then, for workloads
that start at a non-zero offset, prefix_ik [P,128], prefix_kv [P,512] and the
raw window rows that precede the chunk, prefix_win [min(W-1, off0), 512].
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

H_I = 64      # indexer heads
D_I = 128     # indexer head dim
H = 64        # attention query heads
D = 512       # shared KV row dim
RATIO = 4


@dataclass
class Workload:
    name: str
    seed: int
    chunks: list          # chunk lengths, in order
    off0: int             # absolute position of the first chunk's first token
    prefix_pooled: int    # synthetic pooled rows already in the cache at off0
    index_topk: int
    window: int
    ratio: int = RATIO
    sample_rows: int = 0  # oracle rows to check per chunk at full size (0 = all)
    tile_rows: tuple = ()  # indexer tile sizes the workload is run with
    t: dict = field(default_factory=dict)

    @property
    def total(self) -> int:
        return sum(self.chunks)

    @property
    def end(self) -> int:
        return self.off0 + self.total

    def chunk_bounds(self):
        """Yield (chunk_index, local_start, T, absolute_offset)."""
        s = 0
        for c, T in enumerate(self.chunks):
            yield c, s, T, self.off0 + s
            s += T


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def draw(w: Workload) -> Workload:
    """Fill ``w.t`` with the workload's tensors (CPU)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    L = w.total
    t = {}
    t["raw_ik"] = _bf16(torch.randn(L, D_I, generator=g))
    t["raw_kv"] = _bf16(torch.randn(L, D, generator=g))
    t["q_idx"] = _bf16(torch.randn(L, H_I, D_I, generator=g))
    t["w"] = torch.randn(L, H_I, generator=g) * 0.125
    t["q"] = _bf16(torch.randn(L, H, D, generator=g))
    P = w.prefix_pooled
    n_win = min(w.window - 1, w.off0)
    if w.off0 > 0:
        t["prefix_ik"] = _bf16(torch.randn(P, D_I, generator=g))
        t["prefix_kv"] = _bf16(torch.randn(P, D, generator=g))
        t["prefix_win"] = _bf16(torch.randn(n_win, D, generator=g))
    else:
        t["prefix_ik"] = torch.zeros(0, D_I, dtype=torch.bfloat16)
        t["prefix_kv"] = torch.zeros(0, D, dtype=torch.bfloat16)
        t["prefix_win"] = torch.zeros(0, D, dtype=torch.bfloat16)
    w.t = t
    return w


def workload(name: str) -> Workload:
    """A named workload (without tensors; call ``draw``)."""
    if name == "zero_prefix_512":
        return Workload(name, 0, [512], 0, 0, index_topk=64, window=128,
                        tile_rows=(512, 192))
    if name == "two_chunks_4098":
        # a 4,098-token prompt in two chunks: [0,2048) then [2048,4098)
        return Workload(name, 1, [2048, 2050], 0, 0, index_topk=512, window=128,
                        tile_rows=(2048, 512))
    if name == "prompt_16k":
        return Workload(name, 2, [2048] * 8, 0, 0, index_topk=2048, window=128,
                        tile_rows=(2048, 512))
    if name == "ctx_128k":
        off = 131072 - 4096
        return Workload(name, 3, [4096], off, off // RATIO, index_topk=2048,
                        window=128, sample_rows=256, tile_rows=(4096, 1024))
    if name == "ctx_1m":
        off = 1048576 - 4096
        return Workload(name, 4, [4096], off, off // RATIO, index_topk=2048,
                        window=128, sample_rows=128, tile_rows=(1024, 4096))
    # compressed attention (ratio 128): every visible pooled row plus the window
    if name == "compressed_16k":
        return Workload(name, 5, [2048] * 8, 0, 0, index_topk=128, window=128, ratio=128,
                        sample_rows=64, tile_rows=(2048,))
    if name == "compressed_128k":
        off = 131072 - 4096
        return Workload(name, 6, [4096], off, off // 128, index_topk=1024, window=128,
                        ratio=128, sample_rows=128, tile_rows=(4096,))
    # the short shapes: an exact 4-row band and a single-row decode step at 128K
    if name == "band_128k":
        off = 131072 - 4
        return Workload(name, 7, [4], off, off // RATIO, index_topk=2048, window=128,
                        tile_rows=(4,))
    if name == "decode_128k":
        off = 131072 - 4
        return Workload(name, 8, [1], off, off // RATIO, index_topk=2048, window=128,
                        tile_rows=(1,))
    raise KeyError(name)


WORKLOADS = ("zero_prefix_512", "two_chunks_4098", "prompt_16k", "ctx_128k", "ctx_1m")
COMPRESSED_WORKLOADS = ("compressed_16k", "compressed_128k")
SHORT_WORKLOADS = ("band_128k", "decode_128k")


def small(seed: int, chunks, index_topk: int, window: int = 128, off0: int = 0,
          prefix_pooled: int = 0, name: str = "small", ratio: int = RATIO) -> Workload:
    """A custom small workload with the same distributions."""
    return Workload(name, seed, list(chunks), off0, prefix_pooled,
                    index_topk=index_topk, window=window, ratio=ratio)


def sample_rows(T: int, S: int):
    """Evenly spaced local rows floor(s*(T-1)/(S-1)), s=0..S-1 (all rows if S<=0 or S>=T)."""
    if S <= 0 or S >= T:
        return list(range(T))
    return sorted(set((s * (T - 1)) // (S - 1) for s in range(S)))
