"""Every write stays inside its buffer, on tiny and ragged shapes: each output the
library writes (pooled cache rows, remainder rows, score scratch, selection,
attention output) sits between two runs of canary words, and the pooled rows past
the append are canaries too; after the calls every canary must be intact. This
stands in for a memory checker (closed on this pool) over the edges where an
off-by-one would land: ragged last tiles, rows that end mid-piece, single-row
chunks, the split attention, the skip path and the long-row top-k."""
import math

import numpy as np
import pytest
import torch

from deepseek_v4_sparse_ratio_gb300 import _binding as B
from deepseek_v4_sparse_ratio_gb300 import inputs

pytestmark = pytest.mark.gpu

GUARD = 4096          # elements on each side: a multiple of 16 bytes for every dtype here
CANARY16 = 0x7A7B     # bf16 buffers (as int16 bits)
CANARY32 = 0x7A7B7C7D  # int32 and fp32 buffers (as int32 bits)


class Guarded:
    """A device buffer of `shape` with GUARD canary elements before and after it."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape))
        self.n = n
        self.buf = torch.empty(GUARD + n + GUARD, dtype=dtype, device="cuda")
        self.bits().fill_(CANARY16 if dtype == torch.bfloat16 else CANARY32)
        self.t = self.buf[GUARD:GUARD + n].view(*shape)

    def bits(self, x=None):
        x = self.buf if x is None else x
        return x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32)

    def canary(self):
        return CANARY16 if self.buf.dtype == torch.bfloat16 else CANARY32

    def check(self, what):
        torch.cuda.synchronize()
        b = self.bits().cpu()
        c = self.canary()
        assert bool((b[:GUARD] == c).all()), f"{what}: write before the buffer"
        assert bool((b[GUARD + self.n:] == c).all()), f"{what}: write past the buffer"


def _state(cap, ratio=4):
    """A PoolState whose four buffers are guarded (its own tensors are replaced)."""
    st = B.PoolState(cap, "cuda", ratio)
    g = {"pooled_kv": Guarded((cap, B.DIM), torch.bfloat16),
         "pooled_ik": Guarded((cap, B.INDEX_DIM), torch.bfloat16),
         "rem_kv": Guarded((ratio - 1, B.DIM), torch.bfloat16),
         "rem_ik": Guarded((ratio - 1, B.INDEX_DIM), torch.bfloat16)}
    for name, gb in g.items():
        setattr(st, name, gb.t)
    st.c.pooled_kv, st.c.pooled_ik = g["pooled_kv"].t.data_ptr(), g["pooled_ik"].t.data_ptr()
    st.c.rem_kv, st.c.rem_ik = g["rem_kv"].t.data_ptr(), g["rem_ik"].t.data_ptr()
    return st, g


def _rows_untouched(gb, first_row):
    torch.cuda.synchronize()
    rest = gb.bits(gb.t[first_row:]).cpu()
    return bool((rest == gb.canary()).all())


@pytest.mark.parametrize("ratio,chunks", [(4, [10, 5, 3, 1, 300, 2]), (128, [100, 200, 60, 1])])
def test_pooling_writes_only_new_rows_and_remainder(dsa, ratio, chunks):
    wl = inputs.draw(inputs.small(61, chunks, index_topk=8, ratio=ratio))
    cap = wl.end // ratio + 3
    st, g = _state(cap, ratio)
    raw_kv = Guarded((wl.total, B.DIM), torch.bfloat16)
    raw_ik = Guarded((wl.total, B.INDEX_DIM), torch.bfloat16)
    raw_kv.t.copy_(wl.t["raw_kv"])
    raw_ik.t.copy_(wl.t["raw_ik"])
    for _, s, T, off in wl.chunk_bounds():
        B.dsa_pool_append(st, raw_kv.t[s:s + T], raw_ik.t[s:s + T], T, off)
        for name in ("pooled_kv", "pooled_ik"):
            assert _rows_untouched(g[name], st.n_pooled), f"{name}: row past the append written"
        for gb_name, gb in g.items():
            gb.check(gb_name)
    raw_kv.check("raw_kv (read only)")
    raw_ik.check("raw_ik (read only)")


@pytest.mark.parametrize("off,T,k,tile", [(8188, 37, 100, 16), (1000, 300, 64, 300),
                                          (4096, 1000, 256, 333), (280000, 37, 2048, 16),
                                          (4000, 96, 1024, 32), (131068, 1, 2048, 1)])
def test_score_topk_writes_stay_in_selection_and_scratch(dsa, off, T, k, tile):
    g = torch.Generator().manual_seed(off + T)
    n = (off + T) // 4
    q_idx = torch.randn(T, 64, 128, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(T, 64, generator=g) * 0.125).cuda()
    pik = Guarded((n, 128), torch.bfloat16)
    pik.t.copy_(torch.randn(n, 128, generator=g).to(torch.bfloat16))
    sel = Guarded((T, k), torch.int32)
    nbytes = B.dsa_score_scratch_bytes(min(tile, T), n)
    scratch = Guarded((max(nbytes // 4, 1),), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsa_index_score_topk(q_idx, w, pik.t, n, T, off, 4, k, tile, scratch.t, sel.t, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    sel.check("selection")
    scratch.check("score scratch")
    pik.check("pooled keys (read only)")
    s = sel.t.cpu().numpy()
    assert ((s >= -1) & (s < n)).all()   # every entry written with an index or -1


@pytest.mark.parametrize("off,T,k", [(0, 3, 4), (1000, 67, 64), (131068, 1, 2048),
                                     (5000, 40, 300)])
def test_attention_writes_stay_in_the_output(dsa, off, T, k):
    n = (off + T) // 4
    g = torch.Generator().manual_seed(off + k)
    raw_start = max(0, off - 127)
    raw = Guarded((off + T - raw_start, 512), torch.bfloat16)
    raw.t.copy_(torch.randn(off + T - raw_start, 512, generator=g).to(torch.bfloat16))
    pooled = Guarded((max(n, 1), 512), torch.bfloat16)
    pooled.t.copy_(torch.randn(max(n, 1), 512, generator=g).to(torch.bfloat16))
    q = torch.randn(T, 64, 512, generator=g).to(torch.bfloat16).cuda()
    rng = np.random.default_rng(off)
    sel = np.full((T, k), -1, np.int32)
    for i in range(T):
        nv = min((off + i + 1) // 4, n)
        m = min(nv, k)
        sel[i, :m] = np.sort(rng.choice(nv, size=m, replace=False)) if m else []
    out = Guarded((T, 64, 512), torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsa_window_sparse_attn(q, raw.t, raw_start, pooled.t, n, torch.from_numpy(sel).cuda(), k,
                             T, off, 4, 128, 1.0 / math.sqrt(512), out.t, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    out.check("attention output")
    raw.check("raw KV (read only)")
    pooled.check("pooled KV (read only)")
    assert torch.isfinite(out.t.float()).all()   # every output element written


def test_whole_chunks_write_only_their_outputs(dsa):
    """Two chunks through dsa_prefill_chunk with every buffer guarded: 71 rows on the
    skip path (17 pooled rows <= 40), then 130 rows on the full path (50 pooled rows,
    tiles of 48 + 48 + 34, a 1-token remainder). After the first chunk the selection
    and output rows past its 71 must still be canaries."""
    wl = inputs.draw(inputs.small(62, [71, 130], index_topk=40))
    cap = wl.end // 4 + 2
    st, g = _state(cap)
    T = max(wl.chunks)
    raw_kv = Guarded((wl.total, B.DIM), torch.bfloat16)
    raw_kv.t.copy_(wl.t["raw_kv"])
    raw_ik = Guarded((wl.total, B.INDEX_DIM), torch.bfloat16)
    raw_ik.t.copy_(wl.t["raw_ik"])
    q_idx = Guarded((wl.total, 64, 128), torch.bfloat16)
    q_idx.t.copy_(wl.t["q_idx"])
    w = Guarded((wl.total, 64), torch.float32)
    w.t.copy_(wl.t["w"])
    q = Guarded((wl.total, 64, 512), torch.bfloat16)
    q.t.copy_(wl.t["q"])
    tile = 48
    scratch = Guarded((B.dsa_score_scratch_bytes(tile, cap) // 4,), torch.float32)
    sel = Guarded((T, wl.index_topk), torch.int32)
    out = Guarded((T, 64, 512), torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _, s, Tc, off in wl.chunk_bounds():
        B.dsa_prefill_chunk(st, raw_kv.t, 0, raw_ik.t[s:s + Tc], q_idx.t[s:s + Tc], w.t[s:s + Tc],
                            q.t[s:s + Tc], Tc, off, wl.index_topk, 128, 1.0 / math.sqrt(512), tile,
                            scratch.t, sel.t[:Tc], out.t[:Tc], status)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert _rows_untouched(g["pooled_kv"], st.n_pooled)
        assert _rows_untouched(g["pooled_ik"], st.n_pooled)
        # rows of the selection and output past this chunk's rows are not written
        if Tc < T:
            assert bool((sel.bits(sel.t[Tc:]).cpu() == CANARY32).all())
            assert bool((out.bits(out.t[Tc:]).cpu() == CANARY16).all())
    for name, gb in list(g.items()) + [("scratch", scratch), ("sel", sel), ("out", out),
                                        ("raw_kv", raw_kv), ("raw_ik", raw_ik),
                                        ("q_idx", q_idx), ("w", w), ("q", q)]:
        gb.check(name)
