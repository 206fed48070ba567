"""The algorithmic work that bench.py divides by in its roofline lines, checked
against closed forms and against the figures of the workload definition: score
2.165 TFLOP at 128K context and 17.56 at 1M; attention 1.168 TFLOP for a
4096-row chunk with a 128-row window and index_topk 2048."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from deepseek_v4_sparse_ratio_gb300 import inputs  # noqa: E402


def _sum_floor_quarter(T):
    """sum_{j=1..T} floor(j/4) for T = 4m: 2m^2 - m."""
    assert T % 4 == 0
    m = T // 4
    return 2 * m * m - m


def test_counts_match_closed_forms_for_prefixed_chunks():
    for name in ("ctx_128k", "ctx_1m"):
        wl = inputs.workload(name)
        T, off = wl.chunks[0], wl.off0
        assert off % 4 == 0 and T % 4 == 0
        c = bench.work_counts(wl)
        # n_vis(off + i) = off/4 + floor((i+1)/4), all below n
        vis = T * (off // 4) + _sum_floor_quarter(T)
        assert c["score_flops"] == 2 * 64 * 128 * vis
        assert c["topk_bytes"] == 4 * vis + T * wl.index_topk * 4
        # every row sees the whole 128-row window and more than 2048 pooled rows
        assert c["attn_flops"] == 4 * 64 * 512 * (128 + 2048) * T


def test_counts_match_the_workload_figures():
    c = bench.work_counts(inputs.workload("ctx_128k"))
    assert round(c["score_flops"] / 1e12, 3) == 2.165
    assert round(c["attn_flops"] / 1e12, 3) == 1.168
    c = bench.work_counts(inputs.workload("ctx_1m"))
    assert round(c["score_flops"] / 1e12, 2) == 17.56
    assert round(c["attn_flops"] / 1e12, 3) == 1.168


def test_compressed_attention_counts_every_visible_pooled_row():
    wl = inputs.workload("compressed_128k")
    T, off, r = wl.chunks[0], wl.off0, wl.ratio
    c = bench.work_counts(wl)
    pooled = sum((off + i + 1) // r for i in range(T))   # all <= index_topk = 1024
    assert all((off + i + 1) // r <= wl.index_topk for i in range(T))
    assert c["attn_flops"] == 4 * 64 * 512 * (128 * T + pooled)


def test_both_bench_arms_print_the_same_config():
    wl = inputs.workload("ctx_128k")
    a = bench.run_config(wl, "ctx_128k", 4096, 1)
    b = bench.run_config(wl, bench.WORKLOAD, 4096, 1)
    assert a == b and a["pooled_rows"] == 32768 and a["chunk"] == 4096


def test_launch_counts_match_the_launch_lists():
    """4 kernels a step at 128K (pool, score, top-k, attention: profiles'
    launch list); 4 for the decode step (remainder copy instead of pooling);
    2 per extra indexer tile; 3 on the skip path (pool, fill, attention)."""
    assert bench.step_launches(inputs.workload("ctx_128k"), 4096) == 4
    assert bench.step_launches(inputs.workload("decode_128k"), 1) == 4
    assert bench.step_launches(inputs.workload("ctx_1m"), 1024) == 1 + 8 + 1
    assert bench.step_launches(inputs.workload("compressed_128k"), 4096) == 3


def test_multi_chunk_prompts_count_every_chunk():
    """A multi-chunk prompt's step is the whole prompt. prompt_16k: chunks 1-4 fit
    index_topk (skip path: pool, fill, attention), chunks 5-8 score in one 2048-row
    tile (pool, score, top-k, attention). two_chunks_4098: the first chunk takes the
    skip path; the second (2,050 rows: two 2048-row tiles) scores and leaves a
    2-token remainder."""
    assert bench.step_launches(inputs.workload("prompt_16k"), 2048) == 4 * 3 + 4 * 4
    assert bench.step_launches(inputs.workload("two_chunks_4098"), 2048) == 3 + (1 + 1 + 2 * 2 + 1)
    c = bench.work_counts(inputs.workload("prompt_16k"))
    # scores only on the full-path chunks 5..8: rows t = 8192..16383, n_vis = floor((t+1)/4)
    vis = sum((t + 1) // 4 for t in range(8192, 16384))
    assert c["score_flops"] == 2 * 64 * 128 * vis
    k = 2048
    keys = sum(min(128, t + 1) + min(k, (t + 1) // 4) for t in range(16384))
    assert c["attn_flops"] == 4 * 64 * 512 * keys
