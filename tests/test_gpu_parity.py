"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small cases compare every output; the five named workloads run at full size
in the same launch configuration as the benchmark and compare sampled rows
(evenly spaced, first and last row included) plus the whole pooled-cache
state. Tolerances are in tests/parity.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_sparse_ratio_gb300 import _binding as B
from deepseek_v4_sparse_ratio_gb300 import inputs
from deepseek_v4_sparse_ratio_gb300.runner import DeviceWorkload

from parity import (attention_reference, bf16_to_f64, check_attention, check_scores,
                    check_selection)

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(512)


def _bits(t):
    return oracle.as_bf16_bits(t.cpu())


# --------------------------------------------------------------------------- (a) pooling

@pytest.mark.parametrize("chunks", [[10], [5, 3, 1, 7, 16, 2, 300], [2046, 2052], [1, 1, 1, 1, 1]])
def test_pool_append_bitexact(dsa, chunks):
    wl = inputs.draw(inputs.small(11, chunks, index_topk=8))
    st = B.PoolState(wl.end // 4 + 1)
    ref = oracle.PoolState(4)
    raw_kv, raw_ik = wl.t["raw_kv"].cuda(), wl.t["raw_ik"].cuda()
    for _, s, T, off in wl.chunk_bounds():
        B.dsa_pool_append(st, raw_kv[s:s + T], raw_ik[s:s + T], T, off)
        ref.append(wl.t["raw_ik"][s:s + T], wl.t["raw_kv"][s:s + T], off)
        assert (st.n_pooled, st.n_tokens, st.n_rem) == (ref.n_pooled, ref.n_tokens, ref.n_rem)
        assert st.c.n_pooled_ik == st.c.n_pooled_kv
    torch.cuda.synchronize()
    n = ref.n_pooled
    assert np.array_equal(_bits(st.pooled_kv[:n]), ref.pooled_kv)
    assert np.array_equal(_bits(st.pooled_ik[:n]), ref.pooled_ik)
    assert np.array_equal(_bits(st.rem_kv[:ref.n_rem]), ref.rem_kv)
    assert np.array_equal(_bits(st.rem_ik[:ref.n_rem]), ref.rem_ik)


@pytest.mark.parametrize("ratio", [4, 128])
def test_pool_sum_where_fp32_rounds(dsa, ratio):
    """Columns whose running sum is not exact in fp32: 2^10, then 2^-20, then
    -2^10 (+ zeros) has the exact mean 2^-20 / ratio, but an fp32 running sum
    loses the 2^-20. Other columns mix in random rows. The pooled rows must
    still equal the oracle's exact row-order sum bit for bit."""
    T = 2 * ratio
    g = torch.Generator().manual_seed(ratio)
    kv = torch.randn(T, 512, generator=g)
    ik = torch.randn(T, 128, generator=g)
    for x in (kv, ik):
        cols = x[:, ::3]
        cols[0::ratio] = 2.0 ** 10
        cols[1::ratio] = 2.0 ** -20
        cols[2::ratio] = -(2.0 ** 10)
        cols[3::ratio] = 0.0
    kv, ik = kv.to(torch.bfloat16), ik.to(torch.bfloat16)
    st = B.PoolState(4, ratio=ratio)
    B.dsa_pool_append(st, kv.cuda(), ik.cuda(), T, 0)
    torch.cuda.synchronize()
    ref = oracle.PoolState(ratio)
    ref.append(ik, kv, 0)
    assert st.n_pooled == ref.n_pooled == 2
    got = _bits(st.pooled_kv[:2])
    assert np.array_equal(got, ref.pooled_kv)
    assert np.array_equal(_bits(st.pooled_ik[:2]), ref.pooled_ik)
    # the exact mean survived (an fp32 running sum would give 0 here)
    mean = torch.tensor(2.0 ** -20 / ratio).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
    if ratio == 4:
        assert got[0, 0] == mean


def test_pool_ten_tokens_then_resume(dsa):
    """The pages' example: 10 tokens -> 2 pooled rows + 2 remainder; then resume."""
    wl = inputs.draw(inputs.small(3, [10, 6], index_topk=64))
    st = B.PoolState(8)
    raw_kv, raw_ik = wl.t["raw_kv"].cuda(), wl.t["raw_ik"].cuda()
    B.dsa_pool_append(st, raw_kv[:10], raw_ik[:10], 10, 0)
    assert (st.n_pooled, st.n_rem) == (2, 2)
    B.dsa_pool_append(st, raw_kv[10:], raw_ik[10:], 6, 10)
    assert (st.n_pooled, st.n_rem) == (4, 0)
    ref = oracle.PoolState(4)
    ref.append(wl.t["raw_ik"], wl.t["raw_kv"], 0)
    assert np.array_equal(_bits(st.pooled_kv[:4]), ref.pooled_kv)
    with pytest.raises(B.DsaError):
        B.dsa_pool_append(st, raw_kv[:4], raw_ik[:4], 4, 12)   # wrong offset
    assert st.n_tokens == 16


# --------------------------------------------------------------------------- (b)(c) score/top-k

def _score_case(seed, off, T, k, dup=False):
    P = off // 4
    g = torch.Generator().manual_seed(seed)
    q_idx = torch.randn(T, 64, 128, generator=g).to(torch.bfloat16)
    w = torch.randn(T, 64, generator=g) * 0.125
    n = (off + T) // 4
    pik = torch.randn(n, 128, generator=g).to(torch.bfloat16)
    if dup:   # repeated key rows: exact score ties that top-k must break by index
        pik[1::3] = pik[0:-1:3][: pik[1::3].shape[0]]
    return q_idx, w, pik, n


@pytest.mark.parametrize("off,T,k,tile", [(1000, 300, 64, 300), (0, 512, 64, 512),
                                          (8188, 37, 100, 37), (4096, 1000, 512, 1000)])
def test_scores_and_topk_match_oracle(dsa, off, T, k, tile):
    q_idx, w, pik, n = _score_case(off + T, off, T, k)
    sel = torch.empty(T, k, dtype=torch.int32, device="cuda")
    scratch = torch.empty(B.dsa_score_scratch_bytes(tile, n) // 4, dtype=torch.float32,
                          device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsa_index_score_topk(q_idx.cuda(), w.cuda(), pik.cuda(), n, T, off, 4, k, tile, scratch,
                           sel, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    pos = off + np.arange(T)
    ref_s, mag = oracle.index_scores(q_idx, w.numpy(), pos, pik, n)
    stride = (n + 127) // 128 * 128
    gpu_s = scratch[: T * stride].view(T, stride)[:, :n].cpu().numpy()
    check_scores(gpu_s, ref_s, mag)
    ref_sel = oracle.topk(ref_s, pos, n, 4, k)
    check_selection(sel.cpu().numpy(), ref_sel, pos, n, k, ref_s, mag)


def test_topk_ties_break_toward_lower_index(dsa):
    off, T, k = 2000, 64, 40
    q_idx, w, pik, n = _score_case(5, off, T, k, dup=True)
    sel = torch.empty(T, k, dtype=torch.int32, device="cuda")
    scratch = torch.empty(B.dsa_score_scratch_bytes(T, n) // 4, dtype=torch.float32,
                          device="cuda")
    B.dsa_index_score_topk(q_idx.cuda(), w.cuda(), pik.cuda(), n, T, off, 4, k, T, scratch, sel)
    torch.cuda.synchronize()
    # the top-k decision is made on the GPU's own fp32 scores: replay it exactly
    stride = (n + 127) // 128 * 128
    gpu_s = scratch[: T * stride].view(T, stride)[:, :n].cpu().numpy()
    pos = off + np.arange(T)
    assert np.array_equal(sel.cpu().numpy(), oracle.topk(gpu_s, pos, n, 4, k))


@pytest.mark.parametrize("L,m,k,T", [(4000, 100, 64, 4), (4000, 100, 64, 320),
                                     (4000, 600, 300, 4), (4000, 600, 300, 320),
                                     (4000, 100, 3000, 320), (20000, 100, 64, 4),
                                     (20000, 100, 64, 320), (20000, 600, 300, 4),
                                     (20000, 600, 300, 320), (20000, 100, 1000, 320),
                                     (20000, 100, 3000, 320), (70000, 100, 64, 320),
                                     (70000, 3000, 2048, 4)])
def test_topk_heavy_ties_on_every_selection_path(dsa, L, m, k, T):
    """m pooled rows are one repeated key aligned with every indexer query, so m
    scores are exactly equal and above all others; the rest are ReLU'd random
    dot products, about half of them exactly 0. With k < m the k-th place is
    inside the repeated group, with k = 3000 it is inside the zeros. The cases
    cover every way the top-k finds its threshold: a few candidates ranked
    against each other, a crowded threshold bin (radix select over the
    candidates), and a bin too crowded to collect (radix select over the row),
    on rows of 4,000, 20,000 and 70,000 scores, in tiles of 4 rows (1024-thread
    CTAs) and of 320 rows (256-thread CTAs). Rows of 20,000 emit from the kept-
    index bitmap when the candidates were ranked against each other (the cut
    inside the repeated group keeps its lowest indices there) and fall back to
    the ordered pass after a radix select. Ties must go to the lowest
    indices."""
    g = torch.Generator().manual_seed(L + m + k)
    off = 4 * L
    n = (off + T) // 4
    v = torch.randn(128, generator=g)
    q_idx = v.expand(T, 64, 128).to(torch.bfloat16).contiguous()
    w = torch.rand(T, 64, generator=g) * 0.125 + 0.01
    pik = torch.randn(n, 128, generator=g)
    dup = torch.randperm(L, generator=g)[:m]
    pik[dup] = 8.0 * v / v.norm() * math.sqrt(128)
    pik = pik.to(torch.bfloat16)
    sel = torch.empty(T, k, dtype=torch.int32, device="cuda")
    scratch = torch.empty(B.dsa_score_scratch_bytes(T, n) // 4, dtype=torch.float32,
                          device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsa_index_score_topk(q_idx.cuda(), w.cuda(), pik.cuda(), n, T, off, 4, k, T, scratch,
                           sel, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    stride = (n + 127) // 128 * 128
    gpu_s = scratch[: T * stride].view(T, stride)[:, :n].cpu().numpy()
    for r in range(T):   # the ties are real: one value over the whole repeated group
        assert np.unique(gpu_s[r, dup.numpy()]).size == 1
    pos = off + np.arange(T)
    assert np.array_equal(sel.cpu().numpy(), oracle.topk(gpu_s, pos, n, 4, k))


@pytest.mark.parametrize("off,T,k,tile", [(280000, 37, 2048, 16), (300004, 160, 1000, 160),
                                          (262150, 90, 64, 31)])
def test_long_rows_match_oracle(dsa, off, T, k, tile):
    """Rows over 65,536 pooled rows take the persistent top-k (16-byte loads, one
    1024-thread CTA walking several rows): ragged row lengths (n_vis not a multiple
    of the 128-score pieces), tiles whose rows outnumber the CTAs, scores compared
    element by element and the selection against the oracle on every row."""
    q_idx, w, pik, n = _score_case(off + T + tile, off, T, k)
    assert n > 65536
    sel = torch.full((T, k), 7, dtype=torch.int32, device="cuda")
    scratch = torch.empty(B.dsa_score_scratch_bytes(tile, n) // 4, dtype=torch.float32,
                          device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsa_index_score_topk(q_idx.cuda(), w.cuda(), pik.cuda(), n, T, off, 4, k, tile, scratch,
                           sel, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    pos = off + np.arange(T)
    ref_s, mag = oracle.index_scores(q_idx, w.numpy(), pos, pik, n)
    check_selection(sel.cpu().numpy(), oracle.topk(ref_s, pos, n, 4, k), pos, n, k, ref_s, mag)
    stride = (n + 127) // 128 * 128
    last0 = ((T - 1) // tile) * tile
    gs = scratch[: (T - last0) * stride].view(T - last0, stride)[:, :n].cpu().numpy()
    check_scores(gs, ref_s[last0:], mag[last0:])


@pytest.mark.parametrize("L,m,k,T", [(70000, 30, 64, 320), (70000, 600, 300, 320),
                                     (70000, 1500, 1024, 320), (70000, 100, 3000, 320),
                                     (70000, 3000, 2048, 96), (70000, 5000, 2048, 96)])
def test_long_row_topk_heavy_ties_in_tiles(dsa, L, m, k, T):
    """Heavy-tie rows of 70,000 scores through the persistent long-row top-k, in
    tiles of T/4 rows (each CTA walks several rows). The sample-guided pass ends
    most rows; with 600-3000 equal top scores it keeps the lowest indices of the
    tied ones by a radix select over their indices; with 5000 equal top scores its
    candidates overflow and the plain passes take over (a bin too crowded to
    collect: radix select over the row). Checked against the oracle's top-k of the
    GPU's own scores, exactly, and against a one-tile run."""
    g = torch.Generator().manual_seed(L + m + k + 1)
    off = 4 * L
    n = (off + T) // 4
    v = torch.randn(128, generator=g)
    q_idx = v.expand(T, 64, 128).to(torch.bfloat16).contiguous()
    w = torch.rand(T, 64, generator=g) * 0.125 + 0.01
    pik = torch.randn(n, 128, generator=g)
    dup = torch.randperm(L, generator=g)[:m]
    pik[dup] = 8.0 * v / v.norm() * math.sqrt(128)
    pik = pik.to(torch.bfloat16)
    tile = T // 4
    sel = torch.empty(T, k, dtype=torch.int32, device="cuda")
    scratch = torch.empty(B.dsa_score_scratch_bytes(tile, n) // 4, dtype=torch.float32,
                          device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsa_index_score_topk(q_idx.cuda(), w.cuda(), pik.cuda(), n, T, off, 4, k, tile, scratch,
                           sel, status)
    # the scores of every row for the exact replay, from a one-tile run
    full = torch.empty(B.dsa_score_scratch_bytes(T, n) // 4, dtype=torch.float32, device="cuda")
    sel1 = torch.empty(T, k, dtype=torch.int32, device="cuda")
    B.dsa_index_score_topk(q_idx.cuda(), w.cuda(), pik.cuda(), n, T, off, 4, k, T, full, sel1,
                           status)
    torch.cuda.synchronize()
    assert status.item() == 0
    stride = (n + 127) // 128 * 128
    gpu_s = full[: T * stride].view(T, stride)[:, :n].cpu().numpy()
    pos = off + np.arange(T)
    assert np.array_equal(sel.cpu().numpy(), oracle.topk(gpu_s, pos, n, 4, k))
    assert torch.equal(sel, sel1)


def test_guided_topk_falls_back_when_the_sample_misleads(dsa):
    """Rows of exactly 70,000 scores whose sampled pieces (17 pieces of 128 scores
    at 128 * floor(c * 547 / 17), the guided pass's rule for this length) hold
    the only high scores: the sample places its bin at those scores, but fewer of
    them exist than index_topk, so the k-th largest lies below it and the plain
    passes must finish the row. Every score is a monotone function of one key
    coefficient, so the expected selection is known exactly."""
    L, k, T = 70000, 3000, 4
    off = 4 * L - 1                      # rows t = off..off+3 all see L pooled rows
    n = (off + T) // 4
    assert n == L and all((off + i + 1) // 4 == L for i in range(T))
    g = torch.Generator().manual_seed(70)
    v = torch.randn(128, generator=g)
    unit = v / v.norm()
    alpha = torch.rand(n, generator=g) * 2.0 - 1.0
    pieces, ns = (L + 127) // 128, max(8, min(64, L // 4096))
    for c in range(ns):
        b = (c * pieces // ns) * 128
        alpha[b:b + 128] = 2.0 + 0.001 * torch.arange(128)   # the high scores
    pik = (alpha[:, None] * unit[None, :] * 4.0).to(torch.bfloat16)
    q_idx = v.expand(T, 64, 128).to(torch.bfloat16).contiguous()
    w = torch.rand(T, 64, generator=g) * 0.125 + 0.01
    sel = torch.empty(T, k, dtype=torch.int32, device="cuda")
    scratch = torch.empty(B.dsa_score_scratch_bytes(T, n) // 4, dtype=torch.float32,
                          device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsa_index_score_topk(q_idx.cuda(), w.cuda(), pik.cuda(), n, T, off, 4, k, T, scratch,
                           sel, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    stride = (n + 127) // 128 * 128
    gpu_s = scratch[: T * stride].view(T, stride)[:, :n].cpu().numpy()
    high = np.isin(np.arange(n), np.concatenate(
        [np.arange((c * pieces // ns) * 128, (c * pieces // ns) * 128 + 128) for c in range(ns)]))
    assert high.sum() < k and (gpu_s[:, high].min(axis=1) > gpu_s[:, ~high].max(axis=1)).all()
    pos = off + np.arange(T)
    assert np.array_equal(sel.cpu().numpy(), oracle.topk(gpu_s, pos, n, 4, k))


@pytest.mark.parametrize("tiles", [(1, 7, 64, 333), (512, 1000)])
def test_tile_size_changes_no_index(dsa, tiles):
    off, T, k = 4096, 1000, 256
    q_idx, w, pik, n = _score_case(9, off, T, k)
    args = [t.cuda() for t in (q_idx, w, pik)]
    outs = []
    for tile in tiles:
        sel = torch.empty(T, k, dtype=torch.int32, device="cuda")
        scratch = torch.empty(B.dsa_score_scratch_bytes(tile, n) // 4, dtype=torch.float32,
                              device="cuda")
        B.dsa_index_score_topk(*args, n, T, off, 4, k, tile, scratch, sel)
        outs.append(sel.cpu())
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("off,T,k", [(0, 10, 64), (0, 200, 50), (4000, 96, 1024)])
def test_skip_path_equals_full_path(dsa, off, T, k):
    """0 < n <= k: the skip path's selection equals the oracle's full path."""
    q_idx, w, pik, n = _score_case(13, off, T, k)
    assert 0 < n <= k
    sel = torch.full((T, k), 7, dtype=torch.int32, device="cuda")
    B.dsa_index_score_topk(None, None, None, n, T, off, 4, k, 16, None, sel)
    pos = off + np.arange(T)
    ref, s, _ = oracle.select(q_idx, w.numpy(), pos, pik, n, 4, k, force_full=True)
    assert s is not None
    assert np.array_equal(sel.cpu().numpy(), ref)


def test_empty_pool_selects_nothing(dsa):
    sel = torch.zeros(3, 8, dtype=torch.int32, device="cuda")
    B.dsa_index_score_topk(None, None, None, 0, 3, 0, 4, 8, 3, None, sel)
    assert torch.all(sel.cpu() == -1)


# --------------------------------------------------------------------------- (d) attention

def _attn_case(seed, off, T, n, k, window=128, full_sel=False):
    g = torch.Generator().manual_seed(seed)
    raw_start = max(0, off - window + 1) - 3
    raw_start = max(raw_start, 0)
    raw = torch.randn(off + T - raw_start, 512, generator=g).to(torch.bfloat16)
    pooled = torch.randn(max(n, 1), 512, generator=g).to(torch.bfloat16)
    q = torch.randn(T, 64, 512, generator=g).to(torch.bfloat16)
    rng = np.random.default_rng(seed)
    sel = np.full((T, k), -1, np.int32)
    for i in range(T):
        nv = min((off + i + 1) // 4, n)
        m = min(nv, k)
        pick = np.arange(m) if full_sel else np.sort(rng.choice(nv, size=m, replace=False))
        sel[i, :m] = pick
    return raw_start, raw, pooled, q, sel


# The window is an argument of the call: besides the model's 128, a single-row window,
# windows of one row more than a key block (129) and of several blocks (300, 512), some
# reaching back past token 0. The last two cases have more tokens than twice the SM count,
# so each persistent CTA takes several tokens in turn (the query reload between tokens, and
# the barrier phases carried across tokens of one, two and three key blocks).
@pytest.mark.parametrize("off,T,k,window", [(0, 67, 16, 128), (1000, 130, 64, 128),
                                            (5000, 40, 300, 128), (0, 3, 4, 128),
                                            (2000, 50, 64, 1), (700, 33, 16, 129),
                                            (2000, 70, 64, 300), (100, 40, 8, 512),
                                            (0, 700, 64, 128), (20000, 400, 256, 128)])
def test_attention_matches_oracle(dsa, off, T, k, window):
    n = (off + T) // 4
    raw_start, raw, pooled, q, sel = _attn_case(off + T + k, off, T, n, k, window)
    out = torch.empty(T, 64, 512, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsa_window_sparse_attn(q.cuda(), raw.cuda(), raw_start, pooled.cuda(), n,
                             torch.from_numpy(sel).cuda(), k, T, off, 4, window, SCALE, out,
                             status)
    torch.cuda.synchronize()
    assert status.item() == 0
    ref = oracle.attention(q, off + np.arange(T), raw, raw_start, pooled, n, sel, window, SCALE)
    check_attention(bf16_to_f64(out), ref)


# Selections padded with -1 inside the list, so that whole 128-entry key blocks hold no
# visible key: T = 3 runs the cluster split mode, where such a block is the first one a CTA
# takes for its token; T = 40 runs one CTA per token, where it follows the window block.
@pytest.mark.parametrize("T", [3, 40])
def test_attention_with_empty_key_blocks(dsa, T):
    off, k = 5000, 1024
    n = (off + T) // 4
    raw_start, raw, pooled, q, sel = _attn_case(77 + T, off, T, n, k)
    sel[:, 256:384] = -1
    sel[:, 640:768] = -1
    out = torch.empty(T, 64, 512, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsa_window_sparse_attn(q.cuda(), raw.cuda(), raw_start, pooled.cuda(), n,
                             torch.from_numpy(sel).cuda(), k, T, off, 4, 128, SCALE, out, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    ref = oracle.attention(q, off + np.arange(T), raw, raw_start, pooled, n, sel, 128, SCALE)
    check_attention(bf16_to_f64(out), ref)


def test_attention_reports_bad_index_and_skips_it(dsa):
    off, T, k = 400, 8, 16
    n = (off + T) // 4
    raw_start, raw, pooled, q, sel = _attn_case(3, off, T, n, k)
    bad = sel.copy()
    bad[2, -1] = n + 5          # beyond the pool: skipped, reported
    good = sel.copy()
    good[2, -1] = -1
    outs = []
    for s in (bad, good):
        out = torch.empty(T, 64, 512, dtype=torch.bfloat16, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        B.dsa_window_sparse_attn(q.cuda(), raw.cuda(), raw_start, pooled.cuda(), n,
                                 torch.from_numpy(s).cuda(), k, T, off, 4, 128, SCALE, out, status)
        torch.cuda.synchronize()
        outs.append((out.cpu(), status.item()))
    assert outs[0][1] == B.DSA_ERR_BOUNDS and outs[1][1] == 0
    assert torch.equal(outs[0][0], outs[1][0])


# --------------------------------------------------------------------------- whole path

def _oracle_prefix_state(wl):
    if wl.off0:
        return oracle.PoolState.from_prefix(wl.t["prefix_ik"], wl.t["prefix_kv"], wl.off0,
                                            wl.ratio)
    return oracle.PoolState(wl.ratio)


def _scratch_rows(dw, T, n, rows):
    """GPU scores of chunk-local `rows` still held in the score scratch after a
    chunk: the scratch holds the chunk's last tile (rows [last0, T)); returns
    (positions in `rows` of the rows found there, their scores [m, n])."""
    tile = min(dw.tile_rows, T)
    last0 = ((T - 1) // tile) * tile
    stride = (n + 127) // 128 * 128
    idx = [i for i, r in enumerate(rows) if r >= last0]
    if not idx:
        return idx, None
    local = torch.tensor([rows[i] - last0 for i in idx], device=dw.scratch.device)
    held = dw.scratch[: (T - last0) * stride].view(T - last0, stride)
    return idx, held.index_select(0, local)[:, :n].cpu().numpy()


def run_workload_parity(wl, tile_rows, sample, stats=None, keep=False):
    """Every chunk of the workload through dsa_prefill_chunk, compared with the
    oracle on the chunk-local rows inputs.sample_rows(T, sample) (all rows when
    sample is 0): selection (tie-band rule), the scores of those rows that the
    last tile left in the scratch (element-wise), the attention output (against
    the oracle's attention over the GPU's own selection where the two selections
    differ inside the tie band), and the pooled cache bit for bit. Returns the
    GPU selections, and with keep=True also each chunk's (rows, oracle result)."""
    dw = DeviceWorkload(wl, tile_rows=tile_rows)
    ref_state = _oracle_prefix_state(wl)
    raw_all = torch.cat([wl.t["prefix_win"], wl.t["raw_kv"]], 0)
    stats = {} if stats is None else stats
    sels, kept = [], []
    for c, s, T, off in wl.chunk_bounds():
        dw.run_chunk(c)
        torch.cuda.synchronize()
        dw.check_status()
        rows = inputs.sample_rows(T, sample)
        res = oracle.prefill_chunk(ref_state, wl.t["raw_ik"][s:s + T], wl.t["raw_kv"][s:s + T],
                                   off, wl.t["q_idx"][s:s + T], wl.t["w"][s:s + T].numpy(),
                                   wl.t["q"][s:s + T], raw_all, dw.raw_start, rows,
                                   wl.index_topk, wl.window, SCALE)
        n = res["n"]
        assert dw.state.n_pooled == n == (off + T) // wl.ratio
        gsel = dw.sel[:T].cpu().numpy()
        sels.append(gsel)
        check_selection(gsel[rows], res["sel"], res["pos"], n, wl.index_topk,
                        res["scores"], res["mag"], ratio=wl.ratio, stats=stats)
        if res["scores"] is not None:
            idx, gs = _scratch_rows(dw, T, n, rows)
            if idx:
                check_scores(gs, res["scores"][idx], res["mag"][idx], stats)
                stats["score_rows"] = stats.get("score_rows", 0) + len(idx)
        ref_out = attention_reference(res, gsel[rows], wl.t["q"][s:s + T][rows], raw_all,
                                      dw.raw_start, ref_state.pooled_kv, wl.window, SCALE)
        err = check_attention(bf16_to_f64(dw.out[rows]), ref_out)
        stats["attn_rel_err"] = max(stats.get("attn_rel_err", 0.0), err)
        stats["attn_rows"] = stats.get("attn_rows", 0) + len(rows)
        if keep:
            kept.append((rows, res))
    n = ref_state.n_pooled
    lo = wl.prefix_pooled
    assert np.array_equal(_bits(dw.state.pooled_kv[lo:n]), ref_state.pooled_kv[lo:n])
    assert np.array_equal(_bits(dw.state.pooled_ik[lo:n]), ref_state.pooled_ik[lo:n])
    assert dw.state.n_rem == ref_state.n_rem
    print(f"\n{wl.name} tile {tile_rows}: {stats}")
    return (sels, kept) if keep else sels


@pytest.mark.parametrize("name", ["zero_prefix_512", "two_chunks_4098", "prompt_16k"])
def test_workload_parity(dsa, name):
    wl = inputs.draw(inputs.workload(name))
    sels = run_workload_parity(wl, wl.tile_rows[0], wl.sample_rows)
    for tile in wl.tile_rows[1:]:
        dw = DeviceWorkload(wl, tile_rows=tile)
        for c, s, T, off in wl.chunk_bounds():
            dw.run_chunk(c)
            assert np.array_equal(dw.sel[:T].cpu().numpy(), sels[c]), f"tile {tile} chunk {c}"


@pytest.mark.parametrize("name", ["ctx_128k", "ctx_1m"])
def test_long_context_parity_and_tile_invariance(dsa, name):
    """Full size, the benchmark's launch configuration: sampled rows against the
    oracle, then the other tile size must give the same selection; the scores of
    every sampled row held by the last tile of either run are compared element
    by element (ctx_128k: one 4096-row tile; ctx_1m: rows 3072-4095 of the
    1024-row tiling, then all sampled rows of the 4096-row tile, which spans
    2,048 key blocks in the score kernel's segments)."""
    wl = inputs.draw(inputs.workload(name))
    stats = {}
    sels, kept = run_workload_parity(wl, wl.tile_rows[0], wl.sample_rows, stats, keep=True)
    if wl.tile_rows[0] >= wl.chunks[0]:
        assert stats["score_rows"] == len(kept[0][0])   # one tile: every sampled row
    other = wl.tile_rows[1]
    dw = DeviceWorkload(wl, tile_rows=other)
    dw.run_chunk(0)
    torch.cuda.synchronize()
    dw.check_status()
    assert np.array_equal(dw.sel[:wl.chunks[0]].cpu().numpy(), sels[0]), "tiling changed an index"
    rows, res = kept[0]
    idx, gs = _scratch_rows(dw, wl.chunks[0], res["n"], rows)
    assert idx
    check_scores(gs, res["scores"][idx], res["mag"][idx], stats)
    stats["score_rows"] += len(idx)
    print(f"{name} after tile {other}: {stats}")
