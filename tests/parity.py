"""Comparison rules between the CUDA path and the oracle.

Tolerances (stated by the workload definition of the path):
  - pooled rows, remainder rows, counters: bit-exact;
  - scores: |gpu - ref| <= 1e-3 * max(|ref|, A) where A = sum_h |w_h| ReLU(dot)
    is the size of the summed terms (plain relative error is ill-conditioned
    where positive and negative head terms cancel); masked entries exactly -inf.
    check_scores also counts the scores that pass only because of A (their
    error exceeds 1e-3 * |ref|), so that widening stays visible;
  - selection: bit-exact, except indices whose oracle score lies within
    1e-3 relative (same scale as above) of the row's k-th score;
  - attention: max|err| <= 1e-2 * max|ref| over every compared row. A row whose
    selection differs from the oracle's only inside the top-k tie band attends
    over another, equally correct key set; its reference is the oracle's
    attention over the GPU's own selection (attention_reference), held to the
    same 1e-2.
"""
import numpy as np

SCORE_RTOL = 1e-3
ATTN_RTOL = 1e-2


def check_scores(gpu: np.ndarray, ref: np.ndarray, mag: np.ndarray, stats: dict | None = None):
    """Element-wise score rule; returns the worst err/bound. With `stats`, also
    records how many finite scores were compared and how many of them passed
    only because the bound uses A rather than |ref|."""
    fin = np.isfinite(ref)
    assert np.array_equal(np.isneginf(gpu), ~fin), "mask differs"
    err = np.abs(gpu[fin].astype(np.float64) - ref[fin].astype(np.float64))
    rel = np.abs(ref[fin]).astype(np.float64)
    bound = SCORE_RTOL * np.maximum(rel, mag[fin])
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} scores out of tolerance; worst {(err / bound).max():.3g}"
    if stats is not None:
        stats["compared"] = stats.get("compared", 0) + int(err.size)
        stats["pass_by_mag"] = stats.get("pass_by_mag", 0) + int((err > SCORE_RTOL * rel).sum())
    return float((err / np.maximum(bound, 1e-300)).max()) if err.size else 0.0


def _kth(scores_row: np.ndarray, k: int):
    idx = np.arange(scores_row.size)
    order = np.lexsort((idx, -scores_row.astype(np.float64)))
    return order[k - 1]


def check_selection(gpu_sel: np.ndarray, ref_sel: np.ndarray, pos, n: int, k: int,
                    ref_scores=None, ref_mag=None, ratio: int = 4, stats: dict | None = None):
    """Compare selections row by row; ref_scores/ref_mag [R, n] for the band rule.
    Returns the number of indices that differ inside the tie band; with `stats`,
    also how many of those swaps are in the band only because it uses A."""
    pos = np.asarray(pos)
    n_band = 0
    for r, t in enumerate(pos):
        nv = min((int(t) + 1) // ratio, n)
        g, e = gpu_sel[r], ref_sel[r]
        gv = g[g >= 0]
        # structure: ascending, unique, in range, -1 padded at the end
        assert np.all(np.diff(gv) > 0), f"row {r}: not strictly ascending"
        assert gv.size == 0 or (gv[0] >= 0 and gv[-1] < nv), f"row {r}: index out of range"
        assert np.all(g[gv.size:] == -1), f"row {r}: padding"
        assert gv.size == min(nv, k), f"row {r}: {gv.size} kept, expected {min(nv, k)}"
        if nv <= k or ref_scores is None:
            assert np.array_equal(g, e), f"row {r}: selection differs"
            continue
        s = ref_scores[r, :nv].astype(np.float64)
        a = ref_mag[r, :nv]
        kk = _kth(ref_scores[r, :nv], k)
        band = np.abs(s - s[kk]) <= SCORE_RTOL * max(abs(s[kk]), a[kk])
        gs, es = np.zeros(nv, bool), np.zeros(nv, bool)
        gs[gv] = True
        es[e[e >= 0]] = True
        diff = (gs != es) & ~band
        assert not diff.any(), f"row {r}: {diff.sum()} indices differ outside the tie band"
        swapped = (gs != es) & band
        n_band += int(swapped.sum())
        if stats is not None:
            rel_band = np.abs(s - s[kk]) <= SCORE_RTOL * abs(s[kk])
            stats["band_swaps"] = stats.get("band_swaps", 0) + int(swapped.sum())
            stats["band_swaps_by_mag"] = (stats.get("band_swaps_by_mag", 0)
                                          + int((swapped & ~rel_band).sum()))
    return n_band


def bf16_to_f64(x) -> np.ndarray:
    return x.float().cpu().numpy().astype(np.float64)


def attention_reference(res: dict, gpu_sel_rows: np.ndarray, q_rows, raw_all, raw_start: int,
                        pooled_kv, window: int, scale: float) -> np.ndarray:
    """The oracle's attention for the compared rows, over the GPU's own selection
    where it differs from the oracle's (check_selection must have accepted it).

    `res` is what oracle.prefill_chunk returned for these rows (its "out" is over
    the oracle's selection); q_rows are the rows' attention queries."""
    import oracle
    same = np.all(gpu_sel_rows == res["sel"], axis=1)
    ref = res["out"]
    if same.all():
        return ref
    d = np.nonzero(~same)[0]
    ref = ref.copy()
    q_bits = oracle.as_bf16_bits(q_rows)[d]
    ref[d] = oracle.attention(q_bits, res["pos"][d], raw_all, raw_start, pooled_kv, res["n"],
                              np.ascontiguousarray(gpu_sel_rows[d]), window, scale)
    return ref


def check_attention(gpu_out: np.ndarray, ref: np.ndarray):
    """max|err| <= 1e-2 * max|ref| over every compared row; returns max|err| / max|ref|."""
    scale = np.abs(ref).max()
    err = np.abs(gpu_out - ref).max() if ref.size else 0.0
    assert err <= ATTN_RTOL * scale, f"attention max|err| {err:.3g} > 1e-2 * {scale:.3g}"
    return float(err / scale) if scale > 0 else 0.0
