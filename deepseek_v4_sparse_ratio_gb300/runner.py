"""Run a synthetic workload chunk by chunk through ``dsa_prefill_chunk``.

Holds the device-resident buffers of one workload (raw rows with the window
prefix, indexer queries and weights, attention queries, the PoolingCache, the
score scratch, the selection and the output) and calls the C ABI once per
chunk. Allocation and marshalling only; the arithmetic is in libdsa.so.
"""
from __future__ import annotations

import math

import torch

from . import _binding as B
from .inputs import Workload


class DeviceWorkload:
    def __init__(self, wl: Workload, tile_rows: int | None = None, device="cuda",
                 keep_outputs: bool = False):
        self.wl = wl
        t = wl.t
        dev = torch.device(device)
        self.device = dev
        n_win = t["prefix_win"].shape[0]
        self.raw_start = wl.off0 - n_win
        self.raw_kv = torch.cat([t["prefix_win"], t["raw_kv"]], 0).to(dev).contiguous()
        self.raw_ik = t["raw_ik"].to(dev).contiguous()
        self.q_idx = t["q_idx"].to(dev).contiguous()
        self.w = t["w"].to(dev).contiguous()
        self.q = t["q"].to(dev).contiguous()
        self.cap = wl.end // wl.ratio
        self.prefix_ik = t["prefix_ik"].to(dev) if wl.off0 else None
        self.prefix_kv = t["prefix_kv"].to(dev) if wl.off0 else None
        self.tmax = max(wl.chunks)
        self.k = wl.index_topk
        self.tile_rows = tile_rows or (wl.tile_rows[0] if wl.tile_rows else self.tmax)
        n_final = wl.end // wl.ratio
        nbytes = B.dsa_score_scratch_bytes(min(self.tile_rows, self.tmax), n_final)
        self.scratch = torch.empty(max(nbytes // 4, 1), dtype=torch.float32, device=dev)
        self.sel = torch.empty(self.tmax, self.k, dtype=torch.int32, device=dev)
        self.out = torch.empty(self.tmax, B.HEADS, B.DIM, dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.scale = 1.0 / math.sqrt(B.DIM)
        self.reset()

    def reset(self) -> None:
        """Fresh PoolingCache at the workload's starting offset."""
        if self.wl.off0:
            self.state = B.PoolState.from_prefix(self.prefix_ik, self.prefix_kv, self.wl.off0,
                                                 self.cap, self.device, self.wl.ratio)
        else:
            self.state = B.PoolState(self.cap, self.device, self.wl.ratio)

    def run_chunk(self, c: int, stream=None) -> None:
        _, s, T, off = list(self.wl.chunk_bounds())[c]
        B.dsa_prefill_chunk(self.state, self.raw_kv, self.raw_start, self.raw_ik[s:s + T],
                            self.q_idx[s:s + T], self.w[s:s + T], self.q[s:s + T], T, off,
                            self.k, self.wl.window, self.scale, self.tile_rows, self.scratch,
                            self.sel[:T], self.out[:T], self.status, stream)

    def check_status(self) -> None:
        st = int(self.status.item())
        if st != 0:
            raise B.DsaError(st, "device status")
