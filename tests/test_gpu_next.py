"""Parity of the rows after the main path: compressed attention (ratio 128,
every visible pooled row attended), exact small-T prefill bands, window-only
local attention and single-token decode steps -- all through the same C ABI
and against the same oracle.

"perf(deepseek-v4): skip redundant all-pooled indexer scoring" (review) and
"perf(deepseek_v4): faster exact DeepSeek-V4 prefill" (Summary item 1) route
LocalAttention, CompressedAttention and SparseCompressedAttention through the
one fused kernel; "perf(dflash): add opt-in exact prefill bands" (Summary,
Band selection) runs exact prefill in bands of 1-4 tokens with downshifts at
compressor boundaries.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_sparse_ratio_gb300 import _binding as B
from deepseek_v4_sparse_ratio_gb300 import inputs
from deepseek_v4_sparse_ratio_gb300.runner import DeviceWorkload

from parity import bf16_to_f64, check_attention, check_selection
from test_gpu_parity import run_workload_parity

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(512)


def _bits(t):
    return oracle.as_bf16_bits(t.cpu())


# --------------------------------------------------------------------------- compressed attention

@pytest.mark.parametrize("chunks", [[100, 200, 60, 1000], [127, 1, 128, 300]])
def test_pool_ratio128_bitexact(dsa, chunks):
    wl = inputs.draw(inputs.small(17, chunks, index_topk=8, ratio=128))
    st = B.PoolState(wl.end // 128 + 1, ratio=128)
    ref = oracle.PoolState(128)
    raw_kv, raw_ik = wl.t["raw_kv"].cuda(), wl.t["raw_ik"].cuda()
    for _, s, T, off in wl.chunk_bounds():
        B.dsa_pool_append(st, raw_kv[s:s + T], raw_ik[s:s + T], T, off)
        ref.append(wl.t["raw_ik"][s:s + T], wl.t["raw_kv"][s:s + T], off)
        assert (st.n_pooled, st.n_tokens, st.n_rem) == (ref.n_pooled, ref.n_tokens, ref.n_rem)
    torch.cuda.synchronize()
    n = ref.n_pooled
    assert np.array_equal(_bits(st.pooled_kv[:n]), ref.pooled_kv)
    assert np.array_equal(_bits(st.pooled_ik[:n]), ref.pooled_ik)
    assert np.array_equal(_bits(st.rem_kv[:ref.n_rem]), ref.rem_kv)


@pytest.mark.parametrize("name", inputs.COMPRESSED_WORKLOADS)
def test_compressed_attention_parity(dsa, name):
    wl = inputs.draw(inputs.workload(name))
    run_workload_parity(wl, wl.tile_rows[0], wl.sample_rows)


# --------------------------------------------------------------------------- exact small-T bands

@pytest.mark.parametrize("k", [4, 64])
def test_small_bands_through_compressor_boundaries(dsa, k):
    """Chunks of 1-4 tokens, landing on and across ratio-4 boundaries."""
    rng = np.random.default_rng(7)
    chunks = [int(c) for c in rng.integers(1, 5, size=60)]
    wl = inputs.draw(inputs.small(8, chunks, index_topk=k))
    run_workload_parity(wl, 3, 0)


# --------------------------------------------------------------------------- local attention / decode

def test_window_only_local_attention_at_long_offset(dsa):
    """No pooled rows: the raw window alone (LocalAttention)."""
    off, T = 50000, 37
    g = torch.Generator().manual_seed(31)
    raw_start = off - 127
    raw = torch.randn(off + T - raw_start, 512, generator=g).to(torch.bfloat16)
    q = torch.randn(T, 64, 512, generator=g).to(torch.bfloat16)
    sel = torch.full((T, 8), -1, dtype=torch.int32)
    out = torch.empty(T, 64, 512, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsa_window_sparse_attn(q.cuda(), raw.cuda(), raw_start, None, 0, sel.cuda(), 8, T, off, 4,
                             128, SCALE, out, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    ref = oracle.attention(q, off + np.arange(T), raw, raw_start, np.zeros((1, 512), np.uint16), 0,
                           sel.numpy(), 128, SCALE)
    check_attention(bf16_to_f64(out), ref)


@pytest.mark.parametrize("name", inputs.SHORT_WORKLOADS)
def test_short_shapes_at_128k_parity(dsa, name):
    """A 4-row band and a 1-row decode step over a 32,767-row pooled prefix: the
    full score + top-k path (n > index_topk) on every row."""
    wl = inputs.draw(inputs.workload(name))
    run_workload_parity(wl, wl.tile_rows[0], 0)


def test_single_token_decode_steps_after_prefill(dsa):
    """A 1000-token prefill, then eight one-token steps (the decode shape)."""
    chunks = [1000] + [1] * 8
    wl = inputs.draw(inputs.small(41, chunks, index_topk=64))
    run_workload_parity(wl, 1000, 0)
