"""The comparison rules of the GPU parity tests, checked on CPU: each rule must
accept the oracle's own results, reject a planted mistake (a wrong score, a
lost mask, an index swapped outside the top-k tie band, broken ordering or
padding, an attention output off by more than the tolerance), and accept the
differences the rules allow (a swap inside the tie band). Mistakes are planted
in copies of oracle results; nothing here runs the CUDA path."""
import numpy as np
import pytest
import torch

import oracle
from parity import check_attention, check_scores, check_selection


def _case(seed=3, off=4000, T=6, k=64):
    g = torch.Generator().manual_seed(seed)
    n = (off + T) // 4
    q_idx = torch.randn(T, 64, 128, generator=g).to(torch.bfloat16)
    w = (torch.randn(T, 64, generator=g) * 0.125).numpy()
    pik = torch.randn(n, 128, generator=g).to(torch.bfloat16)
    pos = off + np.arange(T)
    s, mag = oracle.index_scores(q_idx, w, pos, pik, n)
    sel = oracle.topk(s, pos, n, 4, k)
    return s, mag, sel, pos, n, k


def test_scores_rule():
    s, mag, _, _, _, _ = _case()
    assert check_scores(s.copy(), s, mag) == 0.0
    bad = s.copy()
    j = int(np.argmax(np.isfinite(bad[0])))
    bad[0, j] += 0.01 * max(abs(s[0, j]), mag[0, j]) + 1e-6   # 10x the tolerance
    with pytest.raises(AssertionError):
        check_scores(bad, s, mag)
    near = s.copy()
    near[0, j] = np.float32(s[0, j] + 1e-4 * max(abs(s[0, j]), mag[0, j]))  # inside
    check_scores(near, s, mag)
    unmasked = s.copy()
    unmasked[-1, -1] = 0.0 if np.isneginf(s[-1, -1]) else -np.inf
    with pytest.raises(AssertionError):
        check_scores(unmasked, s, mag)


def test_selection_rule_rejects_planted_mistakes():
    s, mag, sel, pos, n, k = _case()
    assert check_selection(sel.copy(), sel, pos, n, k, s, mag) == 0
    r = 0
    nv = min((int(pos[r]) + 1) // 4, n)
    row = s[r, :nv].astype(np.float64)
    order = np.lexsort((np.arange(nv), -row))
    kept, dropped = order[:k], order[k:]
    # swap the best kept index for the worst dropped one: far outside the band
    wrong = sel.copy()
    keep = set(wrong[r][wrong[r] >= 0].tolist())
    keep.discard(int(kept[0]))
    keep.add(int(dropped[-1]))
    wrong[r, :k] = sorted(keep)
    with pytest.raises(AssertionError):
        check_selection(wrong, sel, pos, n, k, s, mag)
    unsorted = sel.copy()
    unsorted[r, [0, 1]] = unsorted[r, [1, 0]]
    with pytest.raises(AssertionError):
        check_selection(unsorted, sel, pos, n, k, s, mag)
    out_of_range = sel.copy()
    out_of_range[r, k - 1] = nv   # not visible to this row
    with pytest.raises(AssertionError):
        check_selection(out_of_range, sel, pos, n, k, s, mag)


def test_selection_rule_accepts_a_swap_inside_the_tie_band():
    s, mag, sel, pos, n, k = _case()
    r = 1
    nv = min((int(pos[r]) + 1) // 4, n)
    order = np.lexsort((np.arange(nv), -s[r, :nv].astype(np.float64)))
    kth, first_out = int(order[k - 1]), int(order[k])
    # make the first dropped score tie the k-th one in a copy of the reference,
    # then swap them in the "gpu" selection: allowed by the band rule
    s2 = s.copy()
    s2[r, first_out] = s2[r, kth]
    swapped = sel.copy()
    keep = set(swapped[r][swapped[r] >= 0].tolist())
    keep.discard(kth)
    keep.add(first_out)
    swapped[r, :k] = sorted(keep)
    assert check_selection(swapped, sel, pos, n, k, s2, mag) == 2


def test_attention_rule():
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((4, 64, 512))
    scale = np.abs(ref).max()
    assert check_attention(ref.copy(), ref) == 0.0
    near = ref.copy()
    near[2, 5, 7] += 0.009 * scale
    check_attention(near, ref)
    off = ref.copy()
    off[2, 5, 7] += 0.02 * scale
    with pytest.raises(AssertionError):
        check_attention(off, ref)


def test_attention_reference_uses_the_gpu_selection_where_it_differs():
    """A row whose selection differs inside the tie band is compared with the
    oracle's attention over the GPU's own selection, at the same 1e-2; rows whose
    selection agrees keep the oracle's output."""
    import oracle
    from parity import attention_reference
    rng = np.random.default_rng(5)
    T, n, k, off = 3, 40, 8, 200
    pos = off + np.arange(T)
    raw = rng.standard_normal((off + T, 512)).astype(np.float32)
    pooled = rng.standard_normal((n, 512)).astype(np.float32)
    q = rng.standard_normal((T, 64, 512)).astype(np.float32)
    import torch
    raw_t, pooled_t, q_t = (torch.from_numpy(x).to(torch.bfloat16) for x in (raw, pooled, q))
    sel = np.stack([np.sort(rng.choice(n, k, replace=False)) for _ in range(T)]).astype(np.int32)
    res = {"sel": sel, "pos": pos, "n": n,
           "out": oracle.attention(q_t, pos, raw_t, 0, pooled_t, n, sel, 128, 0.04)}
    gsel = sel.copy()
    free = sorted(set(range(n)) - set(sel[1].tolist()))
    gsel[1, 0] = free[0]
    gsel[1] = np.sort(gsel[1])
    ref = attention_reference(res, gsel, q_t, raw_t, 0, pooled_t, 128, 0.04)
    assert np.array_equal(ref[[0, 2]], res["out"][[0, 2]])
    direct = oracle.attention(q_t[1:2], pos[1:2], raw_t, 0, pooled_t, n, gsel[1:2], 128, 0.04)
    assert np.array_equal(ref[1:2], direct)
    assert not np.allclose(ref[1], res["out"][1])
    # the oracle's own output for the differing row would fail the rule
    with pytest.raises(AssertionError):
        check_attention(direct, res["out"][1:2])
