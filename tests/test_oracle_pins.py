"""Pins of the CPU oracle to things other than itself.

Each test checks an oracle function against what the pages fix (the 10-token
example, the score-scratch arithmetic), closed forms, brute force on tiny
inputs, or a library routine the case reduces to (numpy einsum / lexsort,
torch's fp32->bf16 cast, torch CPU scaled_dot_product_attention in fp64).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_sparse_ratio_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")


# --------------------------------------------------------------------------- bf16 rounding

def _bf16_grid():
    """All finite non-negative bf16 values as float64 (sorted) with their bits."""
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # +0 .. largest finite
    vals = (bits << 16).view(np.float32).astype(np.float64)
    return vals, bits.astype(np.uint16)


def _nearest_bf16_bruteforce(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 by search over the whole grid; ties go to the even bit pattern."""
    vals, bits = _bf16_grid()
    ax = np.abs(x)
    hi = np.searchsorted(vals, ax, side="left").clip(1, len(vals) - 1)
    lo = hi - 1
    dlo, dhi = ax - vals[lo], vals[hi] - ax
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (bits[hi] % 2 == 0))
    out = np.where(pick_hi, bits[hi], bits[lo]).astype(np.uint16)
    return np.where(np.signbit(x), out | 0x8000, out).astype(np.uint16)


def test_round_bf16_ties_to_even_examples():
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 0x3F80      # tie -> even (1.0)
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82  # tie -> even (1+2^-6)
    assert oracle.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81  # just above the tie
    assert oracle.round_bf16(-2.5) == 0xC020
    assert oracle.round_bf16(0.0) == 0 and oracle.round_bf16(-0.0) == 0x8000
    assert oracle.round_bf16(3.5e38) == 0x7F80                # overflow to +inf


def test_round_bf16_matches_bruteforce_nearest():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(20000) * np.exp2(rng.integers(-30, 30, 20000))
    # exact midpoints between neighbouring bf16 values, both parities
    vals, _ = _bf16_grid()
    i = rng.integers(1, 0x7F00, 4000)
    mids = (vals[i] + vals[i + 1]) / 2
    x = np.concatenate([x, mids, -mids])
    assert np.array_equal(oracle.round_bf16_array(x), _nearest_bf16_bruteforce(x))


def test_round_bf16_agrees_with_torch_on_fp32_inputs():
    # for fp32 inputs a single RNE step is what torch's fp32->bf16 cast does
    g = torch.Generator().manual_seed(3)
    x32 = torch.randn(50000, generator=g) * 10
    ref = x32.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16_array(x32.double().numpy())
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------- pooling / state

def _bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


def test_ten_token_prefill_example_from_the_pages():
    ex = json.load(open(GOLDEN))["ten_token_prefill"]
    T = ex["tokens"]
    st = oracle.PoolState(ex["ratio"])
    st.append(_bf16((T, 128), 1), _bf16((T, 512), 2), 0)
    assert st.n_pooled == ex["pooled_rows"]
    assert st.n_rem == ex["remainder"]
    assert st.n_tokens == T
    # selection of the last row: skip path (n <= index_topk) gives sequential rows
    pos = np.arange(T)
    qi, w = _bf16((T, 64, 128), 3), torch.randn(T, 64) * 0.125
    sel, s, _ = oracle.select(qi, w.numpy(), pos, st.pooled_ik, st.n_pooled, 4, 64)
    assert s is None  # full scoring path not invoked
    assert list(sel[-1][sel[-1] >= 0]) == ex["last_row_selection"]
    # the full path reaches the same selection
    sel_full, s_full, _ = oracle.select(qi, w.numpy(), pos, st.pooled_ik, st.n_pooled, 4, 64,
                                        force_full=True)
    assert s_full is not None
    assert np.array_equal(sel, sel_full)


def test_pool_is_rounded_exact_mean():
    x = _bf16((64, 40), 11)
    got = oracle.pool_rows(x, 4)
    xs = oracle.bf16_bits_to_f64(oracle.as_bf16_bits(x)).reshape(16, 4, 40)
    mean = (xs[:, 0] + xs[:, 1] + xs[:, 2] + xs[:, 3]) / 4  # exact in fp64 for bf16 inputs
    assert np.array_equal(got, _nearest_bf16_bruteforce(mean))


@pytest.mark.parametrize("ratio", [2, 8, 32, 128])
def test_pool_any_ratio_is_rounded_exact_rational_mean(ratio):
    """Every power-of-two ratio: the exact mean (rational arithmetic, no floating
    sum at all), rounded once to the nearest bf16. Columns 0 and 1 start each group
    with 2^10, 2^-20, -2^10, which a running fp32 sum would round; column 0 then
    holds zeros, so its exact mean is 2^-20 / ratio, column 1 random values."""
    from fractions import Fraction
    x = torch.randn(2 * ratio, 24, generator=torch.Generator().manual_seed(ratio))
    for c in (0, 1):
        x[0::ratio, c], x[1::ratio, c], x[2::ratio, c] = 2.0 ** 10, 2.0 ** -20, -(2.0 ** 10)
    for r in range(3, ratio):
        x[r::ratio, 0] = 0.0
    xs = oracle.bf16_bits_to_f64(oracle.as_bf16_bits(x.to(torch.bfloat16)))
    got = oracle.pool_rows(x.to(torch.bfloat16), ratio)
    mean = np.empty((2, 24))
    for g in range(2):
        for c in range(24):
            m = sum(Fraction(v) for v in xs[g * ratio:(g + 1) * ratio, c]) / ratio
            assert Fraction(float(m)) == m   # representable in fp64: no rounding yet
            mean[g, c] = float(m)
    assert np.array_equal(got, _nearest_bf16_bruteforce(mean))
    if ratio == 2:   # group [2^10, 2^-20]: mean 2^9 + 2^-21 rounds to 2^9
        assert got[0, 0] == _nearest_bf16_bruteforce(np.array([2.0 ** 9]))[0]
    else:            # [2^10, 2^-20, -2^10, 0, ...]: the mean is exactly 2^-20 / ratio
        assert got[0, 0] == _nearest_bf16_bruteforce(np.array([2.0 ** -20 / ratio]))[0]


@pytest.mark.parametrize("ratio", [16, 128])
def test_pool_closed_forms_large_ratio(ratio):
    """n = floor(N/ratio) and rem = N mod ratio after every chunk; chunking changes
    no pooled row."""
    rng = np.random.default_rng(ratio)
    N = 3 * ratio + ratio // 2 + 1
    ik, kv = _bf16((N, 128), 41), _bf16((N, 512), 42)
    one = oracle.PoolState(ratio)
    one.append(ik, kv, 0)
    for trial in range(6):
        cuts = sorted(rng.choice(np.arange(1, N), size=rng.integers(1, 6), replace=False))
        st = oracle.PoolState(ratio)
        prev = 0
        for c in list(cuts) + [N]:
            st.append(ik[prev:c], kv[prev:c], prev)
            assert st.n_pooled == c // ratio and st.n_rem == c % ratio
            prev = c
        assert np.array_equal(st.pooled_ik, one.pooled_ik)
        assert np.array_equal(st.pooled_kv, one.pooled_kv)


def test_pool_closed_forms_and_chunking_invariance():
    rng = np.random.default_rng(5)
    N = 37
    ik, kv = _bf16((N, 128), 21), _bf16((N, 512), 22)
    one = oracle.PoolState(4)
    one.append(ik, kv, 0)
    for trial in range(20):
        cuts = sorted(rng.choice(np.arange(1, N), size=rng.integers(1, 8), replace=False))
        st = oracle.PoolState(4)
        prev = 0
        for c in list(cuts) + [N]:
            st.append(ik[prev:c], kv[prev:c], prev)
            assert st.n_pooled == c // 4 and st.n_rem == c % 4   # closed form after each chunk
            prev = c
        assert np.array_equal(st.pooled_ik, one.pooled_ik)
        assert np.array_equal(st.pooled_kv, one.pooled_kv)
        assert np.array_equal(st.rem_kv, oracle.as_bf16_bits(kv)[N - N % 4:])


def test_offset_mismatch_is_rejected():
    st = oracle.PoolState(4)
    st.append(_bf16((5, 128), 1), _bf16((5, 512), 2), 0)
    with pytest.raises(ValueError):
        st.append(_bf16((3, 128), 1), _bf16((3, 512), 2), 4)


@pytest.mark.parametrize("name", inputs.WORKLOADS + inputs.SHORT_WORKLOADS)
def test_workload_cache_states_closed_form(name):
    """Pooled rows after each chunk: floor(tokens/4); remainder tokens mod 4."""
    wl = inputs.workload(name)
    st = oracle.PoolState(4, dim_ik=1, dim_kv=1)
    if wl.off0:
        P = wl.prefix_pooled
        st = oracle.PoolState.from_prefix(np.zeros((P, 1), np.uint16), np.zeros((P, 1), np.uint16),
                                          wl.off0)
    got = []
    for _, _, T, off in wl.chunk_bounds():
        st.append(np.zeros((T, 1), np.uint16), np.zeros((T, 1), np.uint16), off)
        got.append((st.n_pooled, st.n_rem))
    expect = {
        "zero_prefix_512": [(128, 0)],
        "two_chunks_4098": [(512, 0), (1024, 2)],
        "prompt_16k": [(512 * c, 0) for c in range(1, 9)],
        "ctx_128k": [(32768, 0)],
        "ctx_1m": [(262144, 0)],
        "band_128k": [(32768, 0)],       # 131,068 + 4 tokens
        "decode_128k": [(32767, 1)],     # 131,068 + 1 token: one raw row left over
    }[name]
    assert got == expect


def test_score_scratch_arithmetic_from_the_pages():
    ex = json.load(open(GOLDEN))["score_scratch_1m"]
    n = ex["ctx"] // ex["ratio"]
    assert abs(n - ex["approx_rows"]) <= 2
    gib = ex["chunk"] * n * 4 / 2 ** 30          # fp32 scores, one per (row, pooled row)
    assert abs(gib - ex["approx_scores_gib"]) < 0.01
    assert 1024 * n * 4 == 2 ** 30               # the 1024-row tile bounds it at 1 GiB


# --------------------------------------------------------------------------- indexer scores

def _score_ref_numpy(q, w, pos, k, ratio):
    """Brute force with numpy einsum in fp64."""
    qd = oracle.bf16_bits_to_f64(oracle.as_bf16_bits(q))
    kd = oracle.bf16_bits_to_f64(oracle.as_bf16_bits(k))
    dots = np.einsum("rhd,jd->rhj", qd, kd)
    s = np.einsum("rh,rhj->rj", np.asarray(w, np.float64), np.maximum(dots, 0))
    a = np.einsum("rh,rhj->rj", np.abs(np.asarray(w, np.float64)), np.maximum(dots, 0))
    nv = np.minimum((np.asarray(pos) + 1) // ratio, k.shape[0])
    mask = np.arange(k.shape[0])[None, :] >= nv[:, None]
    return np.where(mask, -np.inf, s), np.where(mask, 0.0, a)


@pytest.mark.parametrize("heads,dim", [(3, 5), (64, 128)])
def test_scores_match_einsum(heads, dim):
    R, n = 7, 9
    q = _bf16((R, heads, dim), 31)
    k = _bf16((n, dim), 32)
    w = (torch.randn(R, heads, generator=torch.Generator().manual_seed(33)) * 0.125).numpy()
    pos = np.array([0, 3, 4, 7, 12, 30, 35])
    s, a = oracle.index_scores(q, w, pos, k, n)
    sr, ar = _score_ref_numpy(q, w, pos, k, 4)
    fin = np.isfinite(sr)
    assert np.array_equal(fin, np.isfinite(s))
    assert np.all(np.isneginf(s[~fin]))
    # one fp32 rounding of an fp64 sum: within half an fp32 ulp plus fp64 noise
    assert np.all(np.abs(s[fin] - sr[fin]) <= np.spacing(np.abs(sr[fin]).astype(np.float32)) * 0.5
                  + 1e-12 * a[fin])
    assert np.allclose(a, ar, rtol=1e-12, atol=0)


def test_scores_one_hot_closed_form():
    """q[t,h] = c_h * e_{p(t,h)} -> dot = c_h * k[j, p(t,h)]: catches any swapped index."""
    R, heads, dim, n = 3, 4, 8, 6
    q = torch.zeros(R, heads, dim)
    c = [1.0, -2.0, 0.5, 4.0]
    p = lambda t, h: (3 * t + 5 * h + 1) % dim
    for t in range(R):
        for h in range(heads):
            q[t, h, p(t, h)] = c[h]
    k = _bf16((n, dim), 41)
    kd = oracle.bf16_bits_to_f64(oracle.as_bf16_bits(k))
    w = np.array([[1.0, 0.25, -0.5, 2.0], [0.5, 1.0, 1.0, -1.0], [2.0, -3.0, 0.125, 1.0]],
                 np.float32)
    pos = np.array([100, 101, 102])
    s, _ = oracle.index_scores(q.to(torch.bfloat16), w, pos, k, n)
    for t in range(R):
        for j in range(n):
            e = sum(float(w[t, h]) * max(0.0, c[h] * kd[j, p(t, h)]) for h in range(heads))
            assert s[t, j] == np.float32(e)


def test_scores_single_head_unit_weight_is_relu_dot():
    q = _bf16((5, 1, 128), 51)
    k = _bf16((4, 128), 52)
    pos = np.full(5, 1000)
    s, _ = oracle.index_scores(q, np.ones((5, 1), np.float32), pos, k, 4)
    ref = np.maximum(oracle.bf16_bits_to_f64(oracle.as_bf16_bits(q))[:, 0, :]
                     @ oracle.bf16_bits_to_f64(oracle.as_bf16_bits(k)).T, 0)
    assert np.allclose(s, ref, rtol=1e-7, atol=0)


def test_score_mask_matches_pooled_causal_closed_form():
    n = 10
    pos = np.arange(0, 44)
    s, _ = oracle.index_scores(_bf16((44, 2, 8), 61), np.ones((44, 2), np.float32), pos,
                               _bf16((n, 8), 62), n)
    for r, t in enumerate(pos):
        visible = min((t + 1) // 4, n)                    # last raw token of row j is 4j+3
        assert np.all(np.isfinite(s[r, :visible]))
        assert np.all(np.isneginf(s[r, visible:]))


# --------------------------------------------------------------------------- top-k

def _topk_lexsort(scores, pos, n, ratio, k):
    out = np.full((len(pos), k), -1, np.int32)
    for r, t in enumerate(pos):
        nv = min((t + 1) // ratio, n)
        idx = np.arange(nv)
        if nv <= k:
            out[r, :nv] = idx
            continue
        order = np.lexsort((idx, -scores[r, :nv].astype(np.float64)))  # score desc, index asc
        out[r] = np.sort(order[:k])
    return out


def test_topk_bruteforce_with_ties():
    rng = np.random.default_rng(9)
    n, k = 300, 17
    pos = np.array([3, 40, 67, 68, 71, 100, 500, 1199, 1200, 5000])
    R = len(pos)
    for scale in (3, 50, 10 ** 6):   # few distinct values -> many ties; then almost none
        s = rng.integers(-scale, scale, (R, n)).astype(np.float32)
        nv = np.minimum((pos + 1) // 4, n)
        s[np.arange(n)[None, :] >= nv[:, None]] = -np.inf
        got = oracle.topk(s, pos, n, 4, k)
        assert np.array_equal(got, _topk_lexsort(s, pos, n, 4, k))


def test_topk_all_equal_keeps_lowest_indices():
    n, k = 50, 8
    s = np.zeros((1, n), np.float32)
    got = oracle.topk(s, np.array([1000]), n, 4, k)
    assert list(got[0]) == list(range(k))


def test_skip_path_equals_full_path():
    rng = np.random.default_rng(4)
    for n, k in [(1, 1), (5, 8), (16, 16), (30, 64)]:
        T = 4 * n + 3
        pos = np.arange(T)
        qi = _bf16((T, 64, 128), int(rng.integers(1 << 30)))
        w = (rng.standard_normal((T, 64)) / 8).astype(np.float32)
        pk = _bf16((n, 128), 5)
        a, sa, _ = oracle.select(qi, w, pos, pk, n, 4, k)
        b, sb, _ = oracle.select(qi, w, pos, pk, n, 4, k, force_full=True)
        assert sa is None and sb is not None
        assert np.array_equal(a, b)


def test_empty_pool_selects_nothing():
    sel, s, _ = oracle.select(_bf16((3, 64, 128), 1), np.ones((3, 64), np.float32),
                              np.arange(3), np.zeros((0, 128), np.uint16), 0, 4, 8)
    assert s is None and np.all(sel == -1)


# --------------------------------------------------------------------------- attention

def _sdpa_ref(q, pos, raw, raw_start, pooled, sel, window, scale):
    """torch CPU fp64 SDPA over [all raw rows ; all pooled rows] with an explicit mask."""
    qd = torch.from_numpy(oracle.bf16_bits_to_f64(oracle.as_bf16_bits(q)))
    keys = np.concatenate([oracle.bf16_bits_to_f64(oracle.as_bf16_bits(raw)),
                           oracle.bf16_bits_to_f64(oracle.as_bf16_bits(pooled))], axis=0)
    kt = torch.from_numpy(keys)
    nr = raw.shape[0]
    R = len(pos)
    mask = torch.zeros(R, keys.shape[0], dtype=torch.bool)
    for r, t in enumerate(pos):
        for u in range(max(0, t - window + 1), t + 1):
            mask[r, u - raw_start] = True
        for j in sel[r]:
            if j >= 0:
                mask[r, nr + j] = True
    out = []
    for r in range(R):
        out.append(torch.nn.functional.scaled_dot_product_attention(
            qd[r:r + 1], kt[None], kt[None], attn_mask=mask[r][None, None], scale=scale)[0])
    return torch.stack(out).numpy()


@pytest.mark.parametrize("n,k", [(6, 8), (0, 4), (6, 3)])
def test_attention_matches_masked_sdpa(n, k):
    heads, dim, window = 3, 16, 5
    T = 30
    raw = _bf16((T, dim), 71)
    pooled = _bf16((max(n, 1), dim), 72)
    q = _bf16((T, heads, dim), 73)
    pos = np.arange(T)
    rng = np.random.default_rng(74)
    sel = np.full((T, k), -1, np.int32)
    for r, t in enumerate(pos):
        nv = min((t + 1) // 4, n)
        pick = np.sort(rng.choice(nv, size=min(nv, k), replace=False)) if nv else []
        sel[r, :len(pick)] = pick
    got = oracle.attention(q, pos, raw, 0, pooled, n, sel, window, 0.3)
    ref = _sdpa_ref(q, pos, raw, 0, pooled[:n] if n else pooled[:0], sel, window, 0.3)
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_attention_single_key_returns_that_row():
    raw = _bf16((1, 512), 81)
    q = _bf16((1, 64, 512), 82)
    out = oracle.attention(q, [0], raw, 0, np.zeros((1, 512), np.uint16), 0,
                           np.full((1, 4), -1, np.int32), 128, 1 / np.sqrt(512))
    ref = oracle.bf16_bits_to_f64(oracle.as_bf16_bits(raw))[0]
    assert np.allclose(out[0], ref[None, :], rtol=0, atol=1e-15)


def test_attention_two_keys_closed_form():
    """Two keys a, b: out = (e^{sa} a + e^{sb} b) / (e^{sa} + e^{sb})."""
    raw = _bf16((2, 8), 91)
    q = _bf16((1, 1, 8), 92)
    out = oracle.attention(q, [1], raw, 0, np.zeros((1, 8), np.uint16), 0,
                           np.full((1, 1), -1, np.int32), 2, 0.7)
    kk = oracle.bf16_bits_to_f64(oracle.as_bf16_bits(raw))
    qq = oracle.bf16_bits_to_f64(oracle.as_bf16_bits(q))[0, 0]
    ea, eb = np.exp(0.7 * qq @ kk[0]), np.exp(0.7 * qq @ kk[1])
    assert np.allclose(out[0, 0], (ea * kk[0] + eb * kk[1]) / (ea + eb), rtol=1e-12)


def test_attention_selection_order_does_not_matter():
    heads, dim = 2, 8
    raw, pooled, q = _bf16((20, dim), 1), _bf16((5, dim), 2), _bf16((1, heads, dim), 3)
    a = oracle.attention(q, [19], raw, 0, pooled, 5, np.array([[0, 1, 2, 3, 4]], np.int32), 4, 0.5)
    b = oracle.attention(q, [19], raw, 0, pooled, 5, np.array([[4, 2, 0, 3, 1]], np.int32), 4, 0.5)
    assert np.allclose(a, b, rtol=1e-13, atol=0)


def test_attention_window_reaches_into_prefix_buffer():
    """raw_start > 0: the window of the chunk's first row reads rows before the chunk."""
    dim = 8
    raw = _bf16((12, dim), 5)
    q = _bf16((1, 1, dim), 6)
    a = oracle.attention(q, [103], raw, 100, np.zeros((1, dim), np.uint16), 0,
                         np.full((1, 1), -1, np.int32), 4, 0.5)
    ref = _sdpa_ref(q, [3], raw, 0, np.zeros((0, dim), np.uint16), [[-1]], 4, 0.5)
    assert np.allclose(a, ref, rtol=1e-12)
    with pytest.raises(ValueError):   # window start 100-... below raw_start
        oracle.attention(q, [102], raw, 100, np.zeros((1, dim), np.uint16), 0,
                         np.full((1, 1), -1, np.int32), 4, 0.5)
