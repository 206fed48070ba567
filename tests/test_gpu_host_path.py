"""dsa_prefill_chunk_host: the whole path from pinned host buffers with the
copies overlapped on a second stream must give exactly what the device path
gives (same kernels, the attention only split into row slices), chunk after
chunk, and leave the PoolingCache in the same state. Its host outputs are also
checked against the oracle directly on 32 evenly spaced rows per chunk."""
import math

import numpy as np
import pytest
import torch

import oracle

from deepseek_v4_sparse_ratio_gb300 import _binding as B
from deepseek_v4_sparse_ratio_gb300 import inputs
from deepseek_v4_sparse_ratio_gb300.runner import DeviceWorkload

from parity import attention_reference, bf16_to_f64, check_attention, check_selection

pytestmark = pytest.mark.gpu


def _small(kind):
    if kind == "skip_then_full":      # 130 rows fit k (skip path), then 70 more do not
        return inputs.small(31, [130, 70], index_topk=40)
    if kind == "decode":              # a prefill, then single-row chunks
        return inputs.small(32, [300, 1, 1, 1], index_topk=16)
    return inputs.workload(kind)


# The host path scores a short first tile (an eighth of a chunk of 1024 rows or more, at
# most tile_rows) before the rest, in tiles of tile_rows: a tile of 200 rows makes the
# first tile and every later one start off a multiple of the tile size. The 4096-row
# chunk at 128K context is the schedule the benchmark times end to end (a 512-row first
# tile, eight attention slices).
@pytest.mark.parametrize("name,copy_stream,tile", [("two_chunks_4098", True, None),
                                                   ("two_chunks_4098", False, None),
                                                   ("two_chunks_4098", True, 200),
                                                   ("ctx_128k", True, None),
                                                   ("skip_then_full", True, None),
                                                   ("decode", True, None)])
def test_host_path_equals_device_path(dsa, name, copy_stream, tile):
    wl = inputs.draw(_small(name))
    if tile:
        wl.tile_rows = (tile,)
    if not wl.tile_rows:
        wl.tile_rows = (64,)
    dw = DeviceWorkload(wl, tile_rows=wl.tile_rows[0])
    W = wl.window
    raw_all = torch.cat([wl.t["prefix_win"], wl.t["raw_kv"]], 0).pin_memory()
    raw_base = wl.off0 - wl.t["prefix_win"].shape[0]
    tmax = max(wl.chunks)
    ws = B.PrefillWorkspace(tmax, wl.index_topk, tmax + W - 1, wl.end // wl.ratio,
                            wl.tile_rows[0])
    if wl.off0:
        st = B.PoolState.from_prefix(wl.t["prefix_ik"].cuda(), wl.t["prefix_kv"].cuda(),
                                     wl.off0, wl.end // wl.ratio, "cuda", wl.ratio)
    else:
        st = B.PoolState(wl.end // wl.ratio, "cuda", wl.ratio)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream() if copy_stream else None
    scale = 1.0 / math.sqrt(B.DIM)
    ref_state = (oracle.PoolState.from_prefix(wl.t["prefix_ik"], wl.t["prefix_kv"], wl.off0,
                                              wl.ratio) if wl.off0 else oracle.PoolState(wl.ratio))
    for c, s, T, off in wl.chunk_bounds():
        dw.run_chunk(c)
        torch.cuda.synchronize()
        dw.check_status()
        r0 = max(0, off - W + 1) - raw_base
        raw_h = raw_all[r0:off + T - raw_base]
        pin = lambda t: t.contiguous().pin_memory()
        sel_h = torch.empty(T, wl.index_topk, dtype=torch.int32).pin_memory()
        out_h = torch.empty(T, B.HEADS, B.DIM, dtype=torch.bfloat16).pin_memory()
        B.dsa_prefill_chunk_host(st, ws, raw_h, raw_base + r0, pin(wl.t["raw_ik"][s:s + T]),
                                 pin(wl.t["q_idx"][s:s + T]), pin(wl.t["w"][s:s + T]),
                                 pin(wl.t["q"][s:s + T]), T, off, wl.index_topk, W, scale,
                                 wl.tile_rows[0], sel_h, out_h, status, None, side)
        torch.cuda.current_stream().synchronize()
        assert status.item() == 0
        assert torch.equal(sel_h, dw.sel[:T].cpu())
        assert torch.equal(out_h.view(torch.int16), dw.out[:T].cpu().view(torch.int16))
        assert (st.n_pooled, st.n_tokens, st.n_rem) == \
            (dw.state.n_pooled, dw.state.n_tokens, dw.state.n_rem)
        rows = inputs.sample_rows(T, 32)
        res = oracle.prefill_chunk(ref_state, wl.t["raw_ik"][s:s + T], wl.t["raw_kv"][s:s + T],
                                   off, wl.t["q_idx"][s:s + T], wl.t["w"][s:s + T].numpy(),
                                   wl.t["q"][s:s + T], raw_all, raw_base, rows, wl.index_topk, W,
                                   scale)
        gsel = sel_h.numpy()[rows]
        check_selection(gsel, res["sel"], res["pos"], res["n"], wl.index_topk, res["scores"],
                        res["mag"], ratio=wl.ratio)
        ref = attention_reference(res, gsel, wl.t["q"][s:s + T][rows], raw_all, raw_base,
                                  ref_state.pooled_kv, W, scale)
        check_attention(bf16_to_f64(out_h[rows]), ref)
    n = st.n_pooled
    assert torch.equal(st.pooled_kv[:n], dw.state.pooled_kv[:n])
    assert torch.equal(st.pooled_ik[:n], dw.state.pooled_ik[:n])
