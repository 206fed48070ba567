// Steps (b) and (c): indexer scores with the pooled-ratio causal mask folded
// into the epilogue, then per-row top-k, in bounded query-row tiles.
//
// "perf(deepseek_v4): faster exact DeepSeek-V4 prefill", Summary item 5 and
// Performance: the DSA indexer scores every causally visible pooled row of
// every query row (linear in context, FLOP-bound), and the pooled-ratio
// causal mask is applied inside the score kernel's epilogue.
// "perf(deepseek-v4): skip redundant all-pooled indexer scoring", Summary:
// when every pooled row fits within index_topk the scoring and top-k are
// skipped and the selection is the sequential indices.
// "[Discussion] Tile indexed-attention scoring independently of the global
// prefill chunk", Possible design: score/top-k run over bounded row tiles that
// reuse one score scratch, so scratch is tile_rows x pooled rows.
//
// Score kernel (tcgen05): s[t,j] = sum_h w[t,h] * ReLU(q[t,h,:] . k[j,:]).
// The contraction is a GEMM with the pooled keys on M (128 rows per MMA) and
// (token, head) pairs on N (4 tokens x 64 heads = 256), K = 128. A persistent
// CTA works through units of (8 tokens, one segment of the key range): it keeps
// the indexer queries of the 8 tokens resident in shared memory (two N=256
// operands) and streams the segment's 128-row key blocks through a TMA ring; the
// accumulators live in TMEM (2 x 256 columns, one per 4-token half), so the
// epilogue thread that owns TMEM lane j holds every head of its tokens for
// pooled row j and reduces them in registers: ReLU, multiply by w, sum over
// heads in order h = 0..63, mask j >= n_vis(t) to -inf, store coalesced.
//
// The epilogue also reduces each row's visible scores to a (min, max) per key
// segment, parked in the row's selection entries until the top-k overwrites them.
//
// Top-k kernel: one CTA per query row. Rows with n_vis <= k keep all visible
// rows. Otherwise 2048 linear bins between the row's min and max (a monotone
// map) locate the bin holding the k-th largest score; that bin's scores are the
// candidates, among which a rank count (or, for a crowded bin, a radix select
// over order-preserving keys) finds the k-th largest value and how many of its
// equals to keep; a final pass in index order emits the kept indices
// ascending, taking equal scores lowest index first.
#include <math.h>

#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace dsa {

namespace {

// ------------------------------------------------------------------ top-k helpers
//
// The helpers below work for a group of NT threads: `tid` is the thread's index
// in the group (the group starts at a warp boundary) and `sync` is the group's
// barrier (the whole CTA here).

constexpr int kBins = 2048;
constexpr int kCandCap = 2048;
constexpr int64_t kBitmapRows = 8192;  // top-k rows from this many scores emit from a bitmap
constexpr uint32_t kNoBin = 0xFFFFFFFFu;  // find_bin found no bin (fewer than `need` counted)

__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t b = __float_as_uint(f);
    return b ^ ((b & 0x80000000u) ? 0xFFFFFFFFu : 0x80000000u);
}

struct CtaSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// Named barrier kId over kThreads threads.
template <int kId, int kThreads>
struct GroupSync {
    __device__ __forceinline__ void operator()() const {
        asm volatile("bar.sync %0, %1;" ::"n"(kId), "n"(kThreads) : "memory");
    }
};

// Shared memory of one top-k group.
template <int NT>
struct TopkShared {
    uint32_t hist[kBins];
    uint32_t cand[kCandCap];
    int32_t cand_j[kCandCap];
    uint32_t warp_sums[NT / 32 + 1];
    uint32_t s_bin, s_above, s_cnt;
    float s_min[NT / 32], s_max[NT / 32];
    uint32_t w_gt[NT / 32], w_eq[NT / 32];
};

// Exclusive group-wide prefix sum of a per-thread value; *total gets the sum.
template <int NT, class Sync>
__device__ __forceinline__ uint32_t group_excl_scan(uint32_t v, int tid, uint32_t *warp_sums,
                                                    uint32_t *total, Sync sync) {
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) warp_sums[warp] = inc;
    sync();
    if (warp == 0) {
        uint32_t x = lane < (NT / 32) ? warp_sums[lane] : 0;
        uint32_t xi = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, xi, o);
            if (lane >= o) xi += y;
        }
        if (lane < (NT / 32)) warp_sums[lane] = xi - x;
        if (lane == (NT / 32) - 1) warp_sums[(NT / 32)] = xi;
    }
    sync();
    const uint32_t r = warp_sums[warp] + inc - v;
    *total = warp_sums[(NT / 32)];
    sync();
    return r;
}

// After hist[0..nb) is filled: the bin b holding the `need`-th largest element
// (counting from the top bin down) and how many elements lie in higher bins.
template <int NT, class Sync>
__device__ __forceinline__ void find_bin(const uint32_t *hist, int nb, uint32_t need, int tid,
                                         uint32_t *warp_sums, uint32_t *s_bin, uint32_t *s_above,
                                         Sync sync) {
    const int per = nb / NT;
    const int top = nb - per * tid;  // thread i owns bins [top-per, top)
    uint32_t mine = 0;
    for (int b = top - per; b < top; ++b) mine += hist[b];
    uint32_t tot;
    uint32_t cum = group_excl_scan<NT>(mine, tid, warp_sums, &tot, sync);
    for (int b = top - 1; b >= top - per; --b) {
        const uint32_t c = hist[b];
        if (cum < need && need <= cum + c) {
            *s_bin = static_cast<uint32_t>(b);
            *s_above = cum;
        }
        cum += c;
    }
    sync();
}

// Radix select over `count` order keys given by key_at(i): the key of the
// need-th largest element and how many elements equal to it are kept
// (11/11/10-bit digits from the top).
template <int NT, class Sync, typename KeyAt>
__device__ __forceinline__ void radix_select(KeyAt key_at, int64_t count, uint32_t need, int tid,
                                             uint32_t *hist, uint32_t *warp_sums, uint32_t *s_bin,
                                             uint32_t *s_above, uint32_t *thr_out,
                                             uint32_t *need_out, Sync sync) {
    uint32_t prefix = 0;
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int bits = pass == 2 ? 10 : 11;
        const int nb = 1 << bits;
        for (int i = tid; i < nb; i += NT) hist[i] = 0;
        sync();
        for (int64_t j = tid; j < count; j += NT) {
            const uint32_t u = key_at(j);
            if (pass == 0 || (u >> (shift + bits)) == prefix)
                atomicAdd(&hist[(u >> shift) & (nb - 1)], 1u);
        }
        sync();
        find_bin<NT>(hist, nb, need, tid, warp_sums, s_bin, s_above, sync);
        prefix = (prefix << bits) | *s_bin;
        need -= *s_above;
        sync();
    }
    *thr_out = prefix;
    *need_out = need;
}

// Per-warp contiguous segments of whole 128-score pieces of one row; within a
// piece lane l holds scores 4l..4l+3 (one 16-byte load). walk() visits the
// warp's segment in index order with U pieces in flight; scores at or beyond hi
// are the visitor's to mask.
template <int NT, int U>
struct RowWalk {
    const float *src;
    int64_t seg, lo, hi;
    int lane;
    __device__ __forceinline__ RowWalk(const float *s, int64_t L, int tid) : src(s), lane(tid & 31) {
        constexpr int NW = NT / 32;
        seg = ((L + NW - 1) / NW + 127) / 128 * 128;
        lo = min(L, seg * (tid >> 5));
        hi = min(L, seg * ((tid >> 5) + 1));
    }
    template <class Visit>
    __device__ __forceinline__ void walk(Visit &&visit, bool last_pass) const {
        for (int64_t base = lo; base < hi; base += 128 * U) {
            float4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t j = base + 128 * u + 4 * lane;
                const float4 *p = reinterpret_cast<const float4 *>(src + j);
                v[u] = j < hi ? (last_pass ? __ldcs(p) : __ldcg(p))
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) visit(base + 128 * u + 4 * lane, v[u]);
        }
    }
};

__device__ __forceinline__ float elem4(const float4 &v, int e) {
    return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// The row's (min, max): from the score kernel's segment ranges parked in
// out[2s], out[2s+1] when nseg > 0, else a pass over the row. Also zeroes the
// histogram and the candidate count.
template <int NT, int U, class Sync>
__device__ __forceinline__ void row_range(const RowWalk<NT, U> &rw, int32_t nseg,
                                          const int32_t *out, TopkShared<NT> &sh, int tid,
                                          Sync sync, float *vmin_out, float *vmax_out) {
    constexpr int NW = NT / 32;
    const int lane = tid & 31, warp = tid >> 5;
    float vmin = INFINITY, vmax = -INFINITY;
    if (nseg > 0) {
        if (warp == 0)
            for (int sg = lane; sg < nseg; sg += 32) {
                vmin = fminf(vmin, __int_as_float(out[2 * sg]));
                vmax = fmaxf(vmax, __int_as_float(out[2 * sg + 1]));
            }
    } else {
        rw.walk([&](int64_t j, const float4 &v) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (j + e < rw.hi) {
                    vmin = fminf(vmin, elem4(v, e));
                    vmax = fmaxf(vmax, elem4(v, e));
                }
        }, false);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        vmin = fminf(vmin, __shfl_xor_sync(0xFFFFFFFFu, vmin, o));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, o));
    }
    if (lane == 0) {
        sh.s_min[warp] = vmin;
        sh.s_max[warp] = vmax;
    }
    for (int i = tid; i < kBins; i += NT) sh.hist[i] = 0;
    if (tid == 0) sh.s_cnt = 0;
    sync();
    vmin = sh.s_min[0];
    vmax = sh.s_max[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) {
        vmin = fminf(vmin, sh.s_min[w]);
        vmax = fmaxf(vmax, sh.s_max[w]);
    }
    *vmin_out = vmin;
    *vmax_out = vmax;
}

// Linear bin of v among kBins between vmin and vmax (a monotone map: every element
// of a higher bin is >= every element of a lower bin).
struct LinearBins {
    float vmin, scale;
    // x = (v - vmin) * scale in [0, kBins]; adding 2^23 leaves round(x) in the low bits of
    // the sum (an FP add and an integer subtract instead of a float-to-int conversion; the
    // rounding is monotone, which is all the bins need)
    __device__ __forceinline__ int operator()(float v) const {
        return min(kBins - 1, __float_as_int(fmaf(v - vmin, scale, 8388608.0f)) - 0x4B000000);
    }
};

// The float whose order key is u (the inverse of order_key).
__device__ __forceinline__ float key_float(uint32_t u) {
    return __uint_as_float((u & 0x80000000u) ? (u ^ 0x80000000u) : ~u);
}

// Emission in index order: kept element j goes to (#above-threshold before j) +
// min(#equal before j, need_eq); w_gt / w_eq hold each warp segment's counts.
template <int NT, int U>
__device__ __forceinline__ void emit_ordered(const RowWalk<NT, U> &rw, uint32_t thr,
                                             uint32_t need_eq, int32_t *out,
                                             const TopkShared<NT> &sh, int tid) {
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t base_gt = 0, base_eq = 0;
    for (int w = 0; w < warp; ++w) {
        base_gt += sh.w_gt[w];
        base_eq += sh.w_eq[w];
    }
    rw.walk([&](int64_t j, const float4 &v) {
        uint32_t gm = 0, em = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (j + e < rw.hi) {
                const uint32_t u = order_key(elem4(v, e));
                gm |= static_cast<uint32_t>(u > thr) << e;
                em |= static_cast<uint32_t>(u == thr) << e;
            }
        // lane-order prefix of (above, equal) counts, packed in 16-bit halves (at
        // most 128 of each per piece)
        const uint32_t mine = static_cast<uint32_t>(__popc(gm)) |
                              (static_cast<uint32_t>(__popc(em)) << 16);
        uint32_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        const uint32_t excl = incl - mine;
        const uint32_t gb = base_gt + (excl & 0xFFFFu), eb = base_eq + (excl >> 16);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t below = (1u << e) - 1u;
            const uint32_t ng = gb + __popc(gm & below), ne = eb + __popc(em & below);
            if ((gm >> e) & 1u) out[ng + min(ne, need_eq)] = static_cast<int32_t>(j + e);
            else if (((em >> e) & 1u) && ne < need_eq) out[ng + ne] = static_cast<int32_t>(j + e);
        }
        const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
        base_gt += tot & 0xFFFFu;
        base_eq += tot >> 16;
    }, true);
}

// After the histogram of the row over `bins` is in sh.hist: find the threshold bin,
// collect its candidates (counting each segment's elements above it), find the exact
// k-th key and its kept equals (candidate rank, radix select over the candidates, or
// over the whole row when the bin overflows), and emit in index order.
template <int NT, int U, class Sync>
__device__ void topk_finish(const RowWalk<NT, U> &rw, int64_t L, int32_t k, LinearBins bin_of,
                            int32_t *__restrict__ out, TopkShared<NT> &sh, int tid, Sync sync) {
    const int lane = tid & 31, warp = tid >> 5;
    find_bin<NT>(sh.hist, kBins, static_cast<uint32_t>(k), tid, sh.warp_sums, &sh.s_bin,
                 &sh.s_above, sync);
    const int bstar = static_cast<int>(sh.s_bin);
    const uint32_t need = static_cast<uint32_t>(k) - sh.s_above;
    uint32_t above = 0;
    rw.walk([&](int64_t j, const float4 &v) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (j + e < rw.hi) {
                const int b = bin_of(elem4(v, e));
                above += b > bstar;
                if (b == bstar) {
                    const uint32_t c = atomicAdd(&sh.s_cnt, 1u);
                    if (c < kCandCap) {
                        sh.cand[c] = order_key(elem4(v, e));
                        sh.cand_j[c] = static_cast<int32_t>(j + e);
                    }
                }
            }
    }, false);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) above += __shfl_xor_sync(0xFFFFFFFFu, above, o);
    if (lane == 0) {
        sh.w_gt[warp] = above;
        sh.w_eq[warp] = 0;
    }
    sync();
    const uint32_t cnt = sh.s_cnt;
    uint32_t thr, need_eq;
    bool counted = false;  // w_gt / w_eq already hold the per-segment counts
    if (cnt <= NT) {
        // few candidates: each thread ranks one against all of them; the need-th
        // largest has fewer than `need` strictly larger keys and at least `need`
        // larger-or-equal ones
        if (static_cast<uint32_t>(tid) < cnt) {
            const uint32_t u = sh.cand[tid];
            uint32_t gt = 0, ge = 0;
            for (uint32_t c = 0; c < cnt; ++c) {
                const uint32_t w = sh.cand[c];
                gt += w > u;
                ge += w >= u;
            }
            if (gt < need && need <= ge) {  // every thread holding that key agrees
                sh.s_bin = u;
                sh.s_above = need - gt;
            }
        }
        sync();
        thr = sh.s_bin;
        need_eq = sh.s_above;
    } else if (cnt <= kCandCap) {
        radix_select<NT>([&](int64_t c) { return sh.cand[c]; }, cnt, need, tid, sh.hist,
                         sh.warp_sums, &sh.s_bin, &sh.s_above, &thr, &need_eq, sync);
    } else {
        radix_select<NT>([&](int64_t j) { return order_key(rw.src[j]); }, L,
                         static_cast<uint32_t>(k), tid, sh.hist, sh.warp_sums, &sh.s_bin,
                         &sh.s_above, &thr, &need_eq, sync);
    }
    if (cnt <= kCandCap) {
        // candidates above / equal to the threshold, by segment
        for (uint32_t c = tid; c < cnt; c += NT) {
            const int w = static_cast<int>(sh.cand_j[c] / rw.seg);
            if (sh.cand[c] > thr) atomicAdd(&sh.w_gt[w], 1u);
            else if (sh.cand[c] == thr) atomicAdd(&sh.w_eq[w], 1u);
        }
        sync();
        counted = true;
    }
    if (!counted) {
        uint32_t ngt = 0, neq = 0;
        rw.walk([&](int64_t j, const float4 &v) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (j + e < rw.hi) {
                    const uint32_t u = order_key(elem4(v, e));
                    ngt += u > thr;
                    neq += u == thr;
                }
        }, false);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            ngt += __shfl_xor_sync(0xFFFFFFFFu, ngt, o);
            neq += __shfl_xor_sync(0xFFFFFFFFu, neq, o);
        }
        if (lane == 0) {
            sh.w_gt[warp] = ngt;
            sh.w_eq[warp] = neq;
        }
        sync();
    }
    emit_ordered<NT, U>(rw, thr, need_eq, out, sh, tid);
}

// Shared memory of the sample-guided pass: the candidates it collects and a bitmap of
// the kept indices of a row of up to kBits scores.
template <int kCap, int kBits>
struct GuidedShared {
    uint32_t key[kCap];
    int32_t idx[kCap];
    uint32_t bitmap[kBits / 32];
    uint32_t cnt, n_eq;
};

// Sample-guided selection of one row (L <= kBits) after its range is known:
//  1. a sample of whole 128-score pieces spread evenly over the row, binned like the
//     row, gives a bin tau that lies, with a wide margin, below the bin of the k-th
//     largest score (the sample's rank k * samples / L plus 3 standard deviations
//     plus 8);
//  2. one pass over the row counts and collects every score in bins >= tau (key,
//     index); the bins below tau are not counted, so most scores cost a compare;
//  3. if the k-th largest lies in a bin >= tau and the candidates fit, it and its
//     kept equals are found exactly among the candidates (radix select); the kept
//     indices are set in a bitmap (ties at the threshold: the lowest indices) and
//     emitted in index order from it, without another pass over the scores.
// Returns 0 when the row is done; 1 when step 3 does not apply (sh.hist then holds
// the row's full histogram, built by one more pass); 2 when the sample cannot place
// tau (sh.hist zeroed).
template <int NT, int U, int kCap, int kBits, class Sync>
__device__ int topk_guided(const RowWalk<NT, U> &rw, int64_t L, int32_t k, LinearBins bin_of,
                           int32_t *__restrict__ out, TopkShared<NT> &sh,
                           GuidedShared<kCap, kBits> &gs, int tid, Sync sync) {
    constexpr int NW = NT / 32;
    const int lane = tid & 31, warp = tid >> 5;
    const int64_t pieces = (L + 127) / 128;
    const int ns = static_cast<int>(max(int64_t{8}, min(int64_t{64}, L / 4096)));
    const int64_t words = (L + 31) / 32;
    for (int64_t w = tid; w < words; w += NT) gs.bitmap[w] = 0;
    if (tid == 0) {
        gs.cnt = 0;
        gs.n_eq = 0;
    }
    // ---- 1. the sample (piece c starts at 128 * floor(c * pieces / ns))
    int64_t samples = 0;
    for (int c = 0; c < ns; ++c) {
        const int64_t base = (c * pieces / ns) * 128;
        samples += min(int64_t{128}, L - base);
        if (c % NW == warp) {
            const int64_t j = base + 4 * lane;
            if (j < L) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(rw.src + j));
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (j + e < L) atomicAdd(&sh.hist[bin_of(elem4(v, e))], 1u);
            }
        }
    }
    sync();
    const double expect = static_cast<double>(k) * static_cast<double>(samples) /
                          static_cast<double>(L);
    const int64_t need_s = static_cast<int64_t>(ceil(expect + 3.0 * sqrt(expect) + 8.0));
    int tau = -1;
    if (need_s < samples) {
        find_bin<NT>(sh.hist, kBins, static_cast<uint32_t>(need_s), tid, sh.warp_sums, &sh.s_bin,
                     &sh.s_above, sync);
        tau = static_cast<int>(sh.s_bin);
    }
    for (int i = tid; i < kBins; i += NT) sh.hist[i] = 0;
    sync();
    if (tau < 0) return 2;
    // ---- 2. the histogram of bins >= tau (only those can hold the k-th largest score if
    // the sample was right, and the bins below are never read then), candidates of the
    // same bins
    rw.walk([&](int64_t j, const float4 &v) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (j + e < rw.hi) {
                const int b = bin_of(elem4(v, e));
                if (b >= tau) {
                    atomicAdd(&sh.hist[b], 1u);
                    const uint32_t c = atomicAdd(&gs.cnt, 1u);
                    if (c < kCap) {
                        gs.key[c] = order_key(elem4(v, e));
                        gs.idx[c] = static_cast<int32_t>(j + e);
                    }
                }
            }
    }, false);
    if (tid == 0) sh.s_bin = kNoBin;  // stays if the bins >= tau hold fewer than k scores
    sync();
    find_bin<NT>(sh.hist, kBins, static_cast<uint32_t>(k), tid, sh.warp_sums, &sh.s_bin,
                 &sh.s_above, sync);
    const uint32_t cnt = gs.cnt;
    if (sh.s_bin == kNoBin || cnt > static_cast<uint32_t>(kCap)) {
        // the sample misled (the k-th largest lies below tau) or the candidates overflow:
        // the full histogram for the plain passes
        for (int i = tid; i < kBins; i += NT) sh.hist[i] = 0;
        sync();
        rw.walk([&](int64_t j, const float4 &v) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (j + e < rw.hi) atomicAdd(&sh.hist[bin_of(elem4(v, e))], 1u);
        }, false);
        sync();
        return 1;
    }
    // ---- 3. every score of the bins >= tau is a candidate, so the k-th largest score
    // overall is the k-th largest candidate
    uint32_t thr, need_eq;
    radix_select<NT>([&](int64_t c) { return gs.key[c]; }, cnt, static_cast<uint32_t>(k), tid,
                     sh.hist, sh.warp_sums, &sh.s_bin, &sh.s_above, &thr, &need_eq, sync);
    uint32_t my_eq = 0;
    for (uint32_t c = tid; c < cnt; c += NT) {
        const uint32_t u = gs.key[c];
        if (u > thr) atomicOr(&gs.bitmap[gs.idx[c] >> 5], 1u << (gs.idx[c] & 31));
        my_eq += u == thr;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) my_eq += __shfl_xor_sync(0xFFFFFFFFu, my_eq, o);
    if (lane == 0 && my_eq) atomicAdd(&gs.n_eq, my_eq);
    sync();
    if (gs.n_eq == need_eq) {
        for (uint32_t c = tid; c < cnt; c += NT)
            if (gs.key[c] == thr) atomicOr(&gs.bitmap[gs.idx[c] >> 5], 1u << (gs.idx[c] & 31));
    } else {
        // more equal keys than kept: the need_eq lowest indices, i.e. the need_eq
        // largest of ~index among the equal keys (other candidates rank below as 0)
        uint32_t cut, one;
        radix_select<NT>(
            [&](int64_t c) {
                return gs.key[c] == thr ? ~static_cast<uint32_t>(gs.idx[c]) : 0u;
            },
            cnt, need_eq, tid, sh.hist, sh.warp_sums, &sh.s_bin, &sh.s_above, &cut, &one, sync);
        for (uint32_t c = tid; c < cnt; c += NT)
            if (gs.key[c] == thr && ~static_cast<uint32_t>(gs.idx[c]) >= cut)
                atomicOr(&gs.bitmap[gs.idx[c] >> 5], 1u << (gs.idx[c] & 31));
    }
    sync();
    // ---- emission in index order from the bitmap: thread t owns a contiguous run of words
    const int64_t per = (words + NT - 1) / NT;
    const int64_t w0 = min(words, per * tid), w1 = min(words, per * (tid + 1));
    uint32_t mine = 0;
    for (int64_t w = w0; w < w1; ++w) mine += __popc(gs.bitmap[w]);
    uint32_t total;
    uint32_t pos = group_excl_scan<NT>(mine, tid, sh.warp_sums, &total, sync);
    for (int64_t w = w0; w < w1; ++w) {
        uint32_t bits = gs.bitmap[w];
        while (bits) {
            const int bit = __ffs(bits) - 1;
            bits &= bits - 1;
            if (pos < static_cast<uint32_t>(k)) out[pos] = static_cast<int32_t>(32 * w + bit);
            ++pos;
        }
    }
    return 0;
}

// Top-k of one score row (L visible scores, L > k) by a group of NT threads with U
// 16-byte loads in flight per thread: the same algorithm as topk_kernel (2048
// linear bins between the row's min and max, the threshold bin's scores as
// candidates, emission of the kept indices in index order). With gs (rows of up to
// kBits scores) the sample-guided pass runs first and usually ends the row after
// one pass over it; otherwise, or when it cannot, the plain passes follow.
template <int NT, int U, int kCap = 1, int kBits = 32, class Sync>
__device__ void topk_row_vec(const float *__restrict__ src, int64_t L, int32_t k, int32_t nseg,
                             int32_t *__restrict__ out, TopkShared<NT> &sh, int tid, Sync sync,
                             GuidedShared<kCap, kBits> *gs = nullptr) {
    const RowWalk<NT, U> rw(src, L, tid);
    float vmin, vmax;
    row_range<NT, U>(rw, nseg, out, sh, tid, sync, &vmin, &vmax);
    if (vmin == vmax) {
        // every visible score is equal: the k lowest indices
        const int warp = tid >> 5;
        if ((tid & 31) == 0) {
            sh.w_gt[warp] = 0;
            sh.w_eq[warp] = static_cast<uint32_t>(rw.hi - rw.lo);
        }
        sync();
        emit_ordered<NT, U>(rw, order_key(vmax), static_cast<uint32_t>(k), out, sh, tid);
        return;
    }
    const LinearBins bin_of{vmin, static_cast<float>(kBins) / (vmax - vmin)};
    if (gs != nullptr && L <= kBits) {
        const int r = topk_guided<NT, U>(rw, L, k, bin_of, out, sh, *gs, tid, sync);
        if (r == 0) return;
        if (r == 1) {
            topk_finish<NT, U>(rw, L, k, bin_of, out, sh, tid, sync);
            return;
        }
    }
    rw.walk([&](int64_t j, const float4 &v) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (j + e < rw.hi) atomicAdd(&sh.hist[bin_of(elem4(v, e))], 1u);
    }, false);
    sync();
    topk_finish<NT, U>(rw, L, k, bin_of, out, sh, tid, sync);
}

// ------------------------------------------------------------------ score kernel

constexpr int kTok = 8;            // query rows per work unit
constexpr int kStages = 2;         // key-block ring depth
constexpr int kEpiWarps = 16;      // one 4-row x 32-lane slice of a TMEM half each
constexpr int kEpiWarp0 = 2;       // warp 0 TMA, warp 1 MMA, warps 2-17 epilogue
constexpr int kScoreThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr uint32_t kBBytes = 2 * 2 * 256 * 128;  // [half][k-chunk][256 rows][128 B]
constexpr uint32_t kAStage = 2 * 128 * 128;      // [k-chunk][128 rows][128 B]
constexpr uint32_t kOffB = 0;
constexpr uint32_t kOffA = kOffB + kBBytes;
constexpr uint32_t kOffW = kOffA + kStages * kAStage;
constexpr uint32_t kOffRng = kOffW + kTok * kHI * 4;  // [16 epilogue warps][4] partial ranges
constexpr uint32_t kOffBar = kOffRng + kEpiWarps * 4 * 4;
constexpr uint32_t kScoreSmem = kOffBar + 256 + 1024;  // + slack for 1024-B alignment
static_assert(kScoreSmem <= 232448, "over the shared memory of one CTA");

struct ScoreParams {
    const float *w;   // [chunk, 64]
    float *scores;    // tile scratch [R, stride]
    int64_t stride;   // floats per scratch row (multiple of 128)
    int64_t n;        // pooled rows
    int64_t offset;   // absolute position of chunk row 0
    int32_t ratio;    // raw tokens per pooled row
    int64_t r0;       // first chunk row of the tile
    int R;            // rows in the tile
    int nseg;         // key-range segments per 8-row group
    int NB;           // stride / 128
    int n_units;      // ceil(R/8) * nseg
    int32_t *rng;     // selection rows [chunk, k] used as range scratch, or null
    int32_t k;        // selection row length
    int32_t *status;
};

struct Unit {
    int row0, nrow, b0, b1, kend;  // MMA over blocks [b0, kend), -inf fill over [kend, b1)
};

__device__ __forceinline__ Unit unit_geom(const ScoreParams &p, int u) {
    Unit x;
    const int g = u / p.nseg, s = u % p.nseg;
    x.row0 = g * kTok;
    x.nrow = min(kTok, p.R - x.row0);
    const int64_t t_last = p.offset + p.r0 + x.row0 + x.nrow - 1;
    const int64_t nv = min(p.n, (t_last + 1) / p.ratio);
    const int kb_vis = static_cast<int>((nv + kScoreBlock - 1) / kScoreBlock);
    x.b0 = static_cast<int>(static_cast<int64_t>(s) * p.NB / p.nseg);
    x.b1 = static_cast<int>(static_cast<int64_t>(s + 1) * p.NB / p.nseg);
    x.kend = max(x.b0, min(x.b1, kb_vis));
    return x;
}

// Wait that ignores the abort flag (used only to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    const uint32_t b = smem_u32(bar);
    const long long t0 = clock64();
    while (!mbar_test(b, parity))
        if (clock64() - t0 > kWaitBudget) break;
}

// Visible pooled rows of tile row `row` (0 past the tile).
__device__ __forceinline__ int64_t row_nvis(const ScoreParams &p, int row) {
    if (row >= p.R) return 0;
    const int64_t t = p.offset + p.r0 + row;
    return min(p.n, (t + 1) / p.ratio);
}

// Stores the masked score of (row, pooled row j) and returns it (-inf when masked
// or when the row is past the tile); nv = row_nvis(p, row), computed once per unit.
__device__ __forceinline__ float store_score(const ScoreParams &p, int row, int64_t nv, int64_t j,
                                             float acc) {
    if (row >= p.R) return -INFINITY;
    // sum of (+0) and (-0) terms can be -0; keep one zero so key order is total
    const float s = j < nv ? (acc == 0.0f ? 0.0f : acc) : -INFINITY;
    __stcs(p.scores + static_cast<int64_t>(row) * p.stride + j, s);
    return s;
}

__global__ void __launch_bounds__(kScoreThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sB = smem + kOffB;
    uint8_t *sA = smem + kOffA;
    float *sW = reinterpret_cast<float *>(smem + kOffW);
    float *sRng = reinterpret_cast<float *>(smem + kOffRng);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *full = bars;                 // [kStages] key block landed
    uint64_t *empty = bars + kStages;      // [kStages] key block consumed by the MMAs
    uint64_t *b_full = bars + 2 * kStages; // queries landed
    uint64_t *b_empty = b_full + 1;        // queries consumed
    uint64_t *t_full = b_full + 2;         // [2] accumulator half ready
    uint64_t *t_empty = b_full + 4;        // [2] accumulator half drained
    uint64_t *drain = b_full + 6;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(b_full + 7);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(b_full, 1);
        mbar_init(b_empty, 1);
        for (int h = 0; h < 2; ++h) {
            mbar_init(&t_full[h], 1);
            mbar_init(&t_empty[h], kEpiWarps);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        const uint64_t pol_k = policy_evict_last();
        const uint64_t pol_q = policy_evict_first();
        int it = 0, bu = 0;
        for (int u = blockIdx.x; u < p.n_units && !*abort_flag; u += gridDim.x) {
            const Unit x = unit_geom(p, u);
            if (x.kend <= x.b0) continue;
            if (!mbar_wait(b_empty, (bu & 1) ^ 1, abort_flag, p.status)) break;
            mbar_expect_tx(b_full, kBBytes);
            const int qrow = static_cast<int>((p.r0 + x.row0) * kHI);
            for (int half = 0; half < 2; ++half)
                for (int kc = 0; kc < 2; ++kc)
                    tma_load_2d(sB + (half * 2 + kc) * 32768, &tm_q, b_full, kc * 64,
                                qrow + half * 256, pol_q);
            ++bu;
            bool ok = true;
            for (int kb = x.b0; kb < x.kend; ++kb) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&full[s], kAStage);
                for (int kc = 0; kc < 2; ++kc)
                    tma_load_2d(sA + s * kAStage + kc * 16384, &tm_k, &full[s], kc * 64,
                                kb * kScoreBlock, pol_k);
                ++it;
            }
            if (!ok) break;
        }
        // make sure no copy into this CTA's shared memory is still in flight
        for (int i = max(0, it - kStages); i < it; ++i)
            drain_wait(&full[i % kStages], (i / kStages) & 1);
        if (bu > 0) drain_wait(b_full, (bu - 1) & 1);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        constexpr uint32_t idesc = idesc_bf16(128, 256, false, false);
        int it = 0, bu = 0, tu0 = 0, tu1 = 0;
        for (int u = blockIdx.x; u < p.n_units && !*abort_flag; u += gridDim.x) {
            const Unit x = unit_geom(p, u);
            if (x.kend <= x.b0) continue;
            if (!mbar_wait(b_full, bu & 1, abort_flag, p.status)) break;
            tc_fence_after();
            ++bu;
            bool ok = true;
            for (int kb = x.b0; kb < x.kend && ok; ++kb) {
                const int s = it % kStages;
                if (!mbar_wait(&full[s], (it / kStages) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int half = 0; half < 2; ++half) {
                    int &tu = half ? tu1 : tu0;
                    if (!mbar_wait(&t_empty[half], (tu & 1) ^ 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + half * 256;
                    for (int kc = 0; kc < 2; ++kc) {
                        const uint64_t ad =
                            desc_sw128(smem_u32(sA + s * kAStage + kc * 16384), 16, 1024);
                        const uint64_t bd =
                            desc_sw128(smem_u32(sB + (half * 2 + kc) * 32768), 16, 1024);
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4)
                            mma_bf16(d, ad + 2 * k4, bd + 2 * k4, idesc, (kc | k4) != 0);
                    }
                    mma_commit(&t_full[half]);
                    ++tu;
                }
                if (!ok) break;
                mma_commit(&empty[s]);
                ++it;
            }
            if (!ok) break;
            mma_commit(b_empty);
        }
        // every MMA issued above must have finished before TMEM is released
        mma_commit(drain);
        drain_wait(drain, 0);
    } else if (warp >= kEpiWarp0) {
        // ---------------- epilogue: 16 warps; warp reads TMEM sub-partition sp = warp % 4
        // (pooled rows j = 32sp .. 32sp+31 of the block) for token tl of each 4-token half
        const int ew = warp - kEpiWarp0;
        const int sp = warp & 3;
        const int tl = ew >> 2;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(sp * 32) << 16);
        const int nthr = 32 * kEpiWarps;
        int tu0 = 0, tu1 = 0;
        // Every epilogue warp walks every unit so that the named barriers
        // below always see all epilogue threads, even after an abort.
        for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
            const Unit x = unit_geom(p, u);
            asm volatile("bar.sync 1, %0;" ::"r"(nthr) : "memory");
            for (int i = ew * 32 + lane; i < kTok * kHI; i += nthr) {
                const int row = x.row0 + i / kHI;
                sW[i] = row < p.R ? __ldg(&p.w[(p.r0 + row) * kHI + (i % kHI)]) : 0.0f;
            }
            asm volatile("bar.sync 1, %0;" ::"r"(nthr) : "memory");
            bool ok = !*abort_flag;
            // once per unit: the compiler left this 64-bit division inside the key-block
            // loop (score + top-k at 128K 1.566 against 1.606 ms with it there)
            const int64_t nv0 = row_nvis(p, x.row0 + tl), nv1 = row_nvis(p, x.row0 + 4 + tl);
            // range of the visible scores of this warp's two rows (half 0 / 1)
            float rmin0 = INFINITY, rmax0 = -INFINITY, rmin1 = INFINITY, rmax1 = -INFINITY;
            for (int kb = x.b0; kb < x.b1 && ok; ++kb) {
                const int64_t j = static_cast<int64_t>(kb) * kScoreBlock + sp * 32 + lane;
                if (kb < x.kend) {
                    for (int half = 0; half < 2; ++half) {
                        int &tu = half ? tu1 : tu0;
                        if (!mbar_wait(&t_full[half], tu & 1, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        ++tu;
                        const int ti = half * 4 + tl;
                        // sum_h w_h * ReLU(v_h): even heads in .x, odd heads in .y of a
                        // packed pair, added at the end (a fixed order for every tile)
                        const float4 *w4 = reinterpret_cast<const float4 *>(sW + ti * kHI);
                        const uint32_t col = half * 256 + tl * 64;
                        uint64_t acc = 0;
                        // both 32-column slices read before one wait, so the accumulator half
                        // is released one TMEM round trip after it is ready (score + top-k at
                        // 128K 1.521 against 1.554 ms with a wait and the first slice's
                        // arithmetic between the two loads)
                        uint32_t va[2][32];
                        tmem_ld32(lane_addr + col, va[0]);
                        tmem_ld32(lane_addr + col + 32, va[1]);
                        tmem_wait_ld();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&t_empty[half]);
#pragma unroll
                        for (int hp = 0; hp < 2; ++hp) {
                            const uint32_t *v = va[hp];
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                // the weights are read here, one 16-byte load per step; the
                                // volatile load keeps the compiler from hoisting all sixteen of
                                // a half ahead of the accumulator's read-out (score + top-k at
                                // 128K: 1.67 against 1.77 ms with them hoisted)
                                float4 ww;
                                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                             : "=f"(ww.x), "=f"(ww.y), "=f"(ww.z), "=f"(ww.w)
                                             : "r"(smem_u32(&w4[8 * hp + q])));
                                uint64_t w01, w23, r01, r23;
                                asm("mov.b64 %0, {%1, %2};" : "=l"(w01) : "f"(ww.x), "f"(ww.y));
                                asm("mov.b64 %0, {%1, %2};" : "=l"(w23) : "f"(ww.z), "f"(ww.w));
                                asm("mov.b64 %0, {%1, %2};"
                                    : "=l"(r01)
                                    : "f"(fmaxf(__uint_as_float(v[4 * q]), 0.0f)),
                                      "f"(fmaxf(__uint_as_float(v[4 * q + 1]), 0.0f)));
                                asm("mov.b64 %0, {%1, %2};"
                                    : "=l"(r23)
                                    : "f"(fmaxf(__uint_as_float(v[4 * q + 2]), 0.0f)),
                                      "f"(fmaxf(__uint_as_float(v[4 * q + 3]), 0.0f)));
                                asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(w01), "l"(r01));
                                asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(w23), "l"(r23));
                            }
                        }
                        float ae, ao;
                        asm("mov.b64 {%0, %1}, %2;" : "=f"(ae), "=f"(ao) : "l"(acc));
                        const float sc = store_score(p, x.row0 + ti, half ? nv1 : nv0, j, ae + ao);
                        const float sv = sc == -INFINITY ? INFINITY : sc;
                        if (half) {
                            rmin1 = fminf(rmin1, sv);
                            rmax1 = fmaxf(rmax1, sc);
                        } else {
                            rmin0 = fminf(rmin0, sv);
                            rmax0 = fmaxf(rmax0, sc);
                        }
                    }
                } else {
                    for (int half = 0; half < 2; ++half)
                        store_score(p, x.row0 + half * 4 + tl, half ? nv1 : nv0, j, -INFINITY);
                }
            }
            if (p.rng) {
                // Each row's (min, max) over this unit's key segment goes to the row's
                // selection entries 2s, 2s+1 (s = segment), so the top-k kernel needs no
                // pass of its own for the range; it overwrites them with the selection.
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    rmin0 = fminf(rmin0, __shfl_xor_sync(0xFFFFFFFFu, rmin0, o));
                    rmax0 = fmaxf(rmax0, __shfl_xor_sync(0xFFFFFFFFu, rmax0, o));
                    rmin1 = fminf(rmin1, __shfl_xor_sync(0xFFFFFFFFu, rmin1, o));
                    rmax1 = fmaxf(rmax1, __shfl_xor_sync(0xFFFFFFFFu, rmax1, o));
                }
                if (lane == 0) {
                    sRng[ew * 4 + 0] = rmin0;
                    sRng[ew * 4 + 1] = rmax0;
                    sRng[ew * 4 + 2] = rmin1;
                    sRng[ew * 4 + 3] = rmax1;
                }
                asm volatile("bar.sync 1, %0;" ::"r"(nthr) : "memory");
                // row ti = 4 * half + tl is held by warps 4tl .. 4tl+3 (one per TMEM lane quarter)
                const int ti = ew * 32 + lane;
                if (ti < kTok && x.row0 + ti < p.R) {
                    const int h = ti >> 2, tq = ti & 3;
                    float mn = INFINITY, mx = -INFINITY;
#pragma unroll
                    for (int e = 4 * tq; e < 4 * tq + 4; ++e) {
                        mn = fminf(mn, sRng[e * 4 + 2 * h]);
                        mx = fmaxf(mx, sRng[e * 4 + 2 * h + 1]);
                    }
                    int32_t *dst = p.rng + (p.r0 + x.row0 + ti) * static_cast<int64_t>(p.k) +
                                   2 * (u % p.nseg);
                    dst[0] = __float_as_int(mn);
                    dst[1] = __float_as_int(mx);
                }
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ top-k kernel

// threads per top-k CTA: 256 (several CTAs per SM) when the tile has rows
// enough to fill the GPU and the rows are short, else 1024
constexpr int kTopkThreads = 256;
constexpr int kTopkThreadsFew = 1024;
constexpr int kTopkThreadsLong = 512;   // persistent CTAs for rows over 64K scores

// One CTA per query row; every pass walks the row in per-warp contiguous
// segments (coalesced, and an ordered last pass emits in index order). With BM,
// rows of kBitmapRows to 32 x kBins scores skip that pass: the kept scores are
// marked in a bitmap while the candidates are collected, and the indices are
// written from it. Rows are taken last first: the score kernel writes the last rows last, so theirs are
// the scores still in L2. With nseg > 0 the row's range comes from the score
// kernel (segment s's min and max in the row's selection entries 2s, 2s+1).
template <int NT, bool BM>
__global__ void __launch_bounds__(NT)
    topk_kernel(const float *__restrict__ scores, int64_t stride, int64_t n, int64_t offset,
                int32_t ratio, int64_t r0, int32_t k, int32_t nseg, int32_t *__restrict__ sel) {
    __shared__ uint32_t hist[kBins];
    __shared__ uint32_t cand[kCandCap];
    __shared__ int32_t cand_j[kCandCap];
    __shared__ uint32_t warp_sums[(NT / 32) + 1];
    __shared__ uint32_t s_bin, s_above, s_cnt;
    __shared__ float s_min[(NT / 32)], s_max[(NT / 32)];
    __shared__ uint32_t w_gt[(NT / 32)], w_eq[(NT / 32)];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row = static_cast<int>(gridDim.x - 1 - blockIdx.x);
    const int64_t t = offset + r0 + row;
    const int64_t L = min(n, (t + 1) / ratio);
    int32_t *out = sel + (r0 + row) * static_cast<int64_t>(k);
    if (L <= k) {
        for (int i = threadIdx.x; i < k; i += NT) out[i] = i < L ? i : -1;
        return;
    }
    const float *src = scores + static_cast<int64_t>(row) * stride;
    const int64_t seg = ((L + (NT / 32) - 1) / (NT / 32) + 31) / 32 * 32;
    const int64_t lo = min(L, seg * warp), hi = min(L, seg * (warp + 1));

    // ---- 1. range of the row
    float vmin = INFINITY, vmax = -INFINITY;
    if (nseg > 0) {
        if (warp == 0)
            for (int sg = lane; sg < nseg; sg += 32) {
                vmin = fminf(vmin, __int_as_float(out[2 * sg]));
                vmax = fmaxf(vmax, __int_as_float(out[2 * sg + 1]));
            }
    } else {
        for (int64_t j = lo + lane; j < hi; j += 32) {
            const float v = src[j];
            vmin = fminf(vmin, v);
            vmax = fmaxf(vmax, v);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        vmin = fminf(vmin, __shfl_xor_sync(0xFFFFFFFFu, vmin, o));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, o));
    }
    if (lane == 0) {
        s_min[warp] = vmin;
        s_max[warp] = vmax;
    }
    for (int i = threadIdx.x; i < kBins; i += NT) hist[i] = 0;
    if (threadIdx.x == 0) s_cnt = 0;
    __syncthreads();
    vmin = s_min[0];
    vmax = s_max[0];
#pragma unroll
    for (int w = 1; w < (NT / 32); ++w) {
        vmin = fminf(vmin, s_min[w]);
        vmax = fmaxf(vmax, s_max[w]);
    }

    uint32_t thr, need_eq;
    bool counted = false;  // w_gt / w_eq already hold the per-segment counts
    if (vmin == vmax) {
        // every visible score is equal: the k lowest indices
        thr = order_key(vmax);
        need_eq = static_cast<uint32_t>(k);
    } else {
        // ---- 2. linear bins between min and max: a monotone map, so every element
        // of a higher bin is >= every element of a lower bin
        const float scale = static_cast<float>(kBins) / (vmax - vmin);
        auto bin_of = [&](float v) {
            return min(kBins - 1, __float_as_int(fmaf(v - vmin, scale, 8388608.0f)) - 0x4B000000);
        };
        // the passes over the row load eight scores per thread before using any of them:
        // one at a time, each pass waited on every load (score + top-k at 128K 1.607
        // against 1.678 ms; four at a time 1.651)
        {
            int64_t j = lo + lane;
            for (; j + 224 < hi; j += 256) {
                float v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = src[j + 32 * q];
#pragma unroll
                for (int q = 0; q < 8; ++q) atomicAdd(&hist[bin_of(v[q])], 1u);
            }
            for (; j < hi; j += 32) atomicAdd(&hist[bin_of(src[j])], 1u);
        }
        __syncthreads();
        find_bin<NT>(hist, kBins, static_cast<uint32_t>(k), threadIdx.x, warp_sums, &s_bin,
                     &s_above, CtaSync{});
        const int bstar = static_cast<int>(s_bin);
        const uint32_t need = static_cast<uint32_t>(k) - s_above;
        // rows of 8K to 64K scores: the histogram's words become the row's kept-index
        // bitmap from here on. Scores above the threshold bin are marked as they are met,
        // the kept candidates after the ranking, and the indices are written from the
        // bitmap, so the row is read twice, not three times (score + top-k at 128K 1.422
        // against 1.493 ms, selections identical). Shorter rows keep the ordered
        // emission pass, and tiles of short rows launch the kernel without this path.
        const bool use_bm = BM && L >= kBitmapRows && L <= static_cast<int64_t>(32) * kBins;
        if (use_bm) {
            for (int i = threadIdx.x; i < static_cast<int>((L + 31) / 32); i += NT) hist[i] = 0;
            __syncthreads();
        }
        // ---- 3. the threshold bin's elements are the candidates; count each
        // segment's elements above that bin on the way
        uint32_t above = 0;
        auto cand_visit = [&](int64_t j, float v) {
            const int b = bin_of(v);
            const bool gt = b > bstar;
            above += gt;
            if (use_bm && gt)
                atomicOr(&hist[static_cast<int>(j) >> 5], 1u << (static_cast<int>(j) & 31));
            if (b == bstar) {
                const uint32_t c = atomicAdd(&s_cnt, 1u);
                if (c < kCandCap) {
                    cand[c] = order_key(v);
                    cand_j[c] = static_cast<int32_t>(j);
                }
            }
        };
        {
            int64_t j = lo + lane;
            for (; j + 224 < hi; j += 256) {
                float v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = src[j + 32 * q];
#pragma unroll
                for (int q = 0; q < 8; ++q) cand_visit(j + 32 * q, v[q]);
            }
            for (; j < hi; j += 32) cand_visit(j, src[j]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) above += __shfl_xor_sync(0xFFFFFFFFu, above, o);
        if (lane == 0) {
            w_gt[warp] = above;
            w_eq[warp] = 0;
        }
        __syncthreads();
        const uint32_t cnt = s_cnt;
        if (cnt <= NT) {
            // few candidates (the usual case: one linear bin near the threshold holds a
            // handful of scores): each thread ranks one candidate against all of them;
            // the need-th largest has fewer than `need` strictly larger keys and at
            // least `need` larger-or-equal ones
            if (threadIdx.x < cnt) {
                const uint32_t u = cand[threadIdx.x];
                uint32_t gt = 0, ge = 0;
                for (uint32_t c = 0; c < cnt; ++c) {
                    const uint32_t v = cand[c];
                    gt += v > u;
                    ge += v >= u;
                }
                if (gt < need && need <= ge) {  // every thread holding that key agrees
                    s_bin = u;
                    s_above = need - gt;
                }
            }
            __syncthreads();
            thr = s_bin;
            need_eq = s_above;
            if (use_bm) {
                // kept candidates: above the threshold key, or equal to it and among the
                // need_eq lowest indices of the equal ones
                if (threadIdx.x < cnt) {
                    const uint32_t u = cand[threadIdx.x];
                    const int32_t jj = cand_j[threadIdx.x];
                    bool keep = u > thr;
                    if (u == thr) {
                        uint32_t before = 0;
                        for (uint32_t c = 0; c < cnt; ++c) before += cand[c] == thr && cand_j[c] < jj;
                        keep = before < need_eq;
                    }
                    if (keep) atomicOr(&hist[jj >> 5], 1u << (jj & 31));
                }
                __syncthreads();
                const int words = static_cast<int>((L + 31) / 32);
                const int per = (words + NT - 1) / NT;
                const int w0 = min(words, per * static_cast<int>(threadIdx.x));
                const int w1 = min(words, w0 + per);
                uint32_t mine = 0;
                for (int w = w0; w < w1; ++w) mine += __popc(hist[w]);
                uint32_t total;
                uint32_t pos = group_excl_scan<NT>(mine, threadIdx.x, warp_sums, &total, CtaSync{});
                for (int w = w0; w < w1; ++w) {
                    uint32_t bits = hist[w];
                    while (bits) {
                        const int bit = __ffs(bits) - 1;
                        out[pos++] = 32 * w + bit;
                        bits &= bits - 1u;
                    }
                }
                return;
            }
        } else if (cnt <= kCandCap) {
            radix_select<NT>([&](int64_t c) { return cand[c]; }, cnt, need, threadIdx.x, hist,
                             warp_sums, &s_bin, &s_above, &thr, &need_eq, CtaSync{});
        }
        if (cnt <= kCandCap) {
            // candidates above / equal to the threshold, by segment
            for (uint32_t c = threadIdx.x; c < cnt; c += NT) {
                const int w = static_cast<int>(cand_j[c] / seg);
                if (cand[c] > thr) atomicAdd(&w_gt[w], 1u);
                else if (cand[c] == thr) atomicAdd(&w_eq[w], 1u);
            }
            __syncthreads();
            counted = true;
        } else {
            radix_select<NT>([&](int64_t j) { return order_key(src[j]); }, L,
                             static_cast<uint32_t>(k), threadIdx.x, hist, warp_sums, &s_bin,
                             &s_above, &thr, &need_eq, CtaSync{});
        }
    }

    // ---- 4. emit kept indices ascending: each warp owns its contiguous segment
    if (!counted) {
        uint32_t ngt = 0, neq = 0;
        for (int64_t base = lo; base < hi; base += 32) {
            const int64_t j = base + lane;
            const uint32_t u = j < hi ? order_key(src[j]) : 0u;
            ngt += __popc(__ballot_sync(0xFFFFFFFFu, j < hi && u > thr));
            neq += __popc(__ballot_sync(0xFFFFFFFFu, j < hi && u == thr));
        }
        if (lane == 0) {
            w_gt[warp] = ngt;
            w_eq[warp] = neq;
        }
        __syncthreads();
    }
    uint32_t base_gt = 0, base_eq = 0;
    for (int w = 0; w < warp; ++w) {
        base_gt += w_gt[w];
        base_eq += w_eq[w];
    }
    const uint32_t lt_mask = (1u << lane) - 1u;
    // the scores hold no -0 (stored as +0) and no NaN, so comparing the values orders
    // them exactly as their keys do (one compare per score instead of its key: score +
    // top-k at 128K 1.554 against 1.566 ms)
    const float t_val = key_float(thr);
    auto emit = [&](int64_t base, float v) {
        const int64_t j = base + lane;
        const bool gt = j < hi && v > t_val;
        const bool eq = j < hi && v == t_val;
        const uint32_t mg = __ballot_sync(0xFFFFFFFFu, gt);
        const uint32_t me = __ballot_sync(0xFFFFFFFFu, eq);
        const uint32_t eq_before = base_eq + __popc(me & lt_mask);
        if (gt || (eq && eq_before < need_eq))
            out[base_gt + __popc(mg & lt_mask) + min(eq_before, need_eq)] = static_cast<int32_t>(j);
        base_gt += __popc(mg);
        base_eq += __popc(me);
    };
    {
        int64_t base = lo;
        for (; base + 224 < hi; base += 256) {
            float v[8];
#pragma unroll
            for (int q = 0; q < 7; ++q) v[q] = src[base + 32 * q + lane];
            v[7] = base + 224 + lane < hi ? src[base + 224 + lane] : 0.0f;
#pragma unroll
            for (int q = 0; q < 8; ++q) emit(base + 32 * q, v[q]);
        }
        for (; base < hi; base += 32) {
            const int64_t j = base + lane;
            emit(base, j < hi ? src[j] : 0.0f);
        }
    }
}

// Long rows: a persistent CTA per SM (or fewer) walks rows R-1-blockIdx.x,
// R-1-blockIdx.x-gridDim.x, ... with 16-byte loads (topk_row_vec). Few rows are in
// flight at once, so the passes after the first find the row in L2.
template <int NT, int U>
__global__ void __launch_bounds__(NT)
    topk_vec_kernel(const float *__restrict__ scores, int64_t stride, int64_t n, int64_t offset,
                    int32_t ratio, int64_t r0, int R, int32_t k, int32_t nseg,
                    int32_t *__restrict__ sel) {
    __shared__ TopkShared<NT> sh;
    for (int it = blockIdx.x; it < R; it += gridDim.x) {
        const int row = R - 1 - it;
        const int64_t t = offset + r0 + row;
        const int64_t L = min(n, (t + 1) / ratio);
        int32_t *out = sel + (r0 + row) * static_cast<int64_t>(k);
        if (L <= k) {
            for (int i = threadIdx.x; i < k; i += NT) out[i] = i < L ? i : -1;
        } else {
            topk_row_vec<NT, U>(scores + static_cast<int64_t>(row) * stride, L, k, nseg, out, sh,
                                threadIdx.x, CtaSync{});
        }
        __syncthreads();  // the shared arrays are reused by the next row
    }
}

// The sample-guided pass in persistent CTAs (as topk_vec_kernel), with its
// candidates and kept-index bitmap in dynamic shared memory: rows of up to kBits
// scores, up to kCap candidates.
template <int NT, int U, int kCap, int kBits>
constexpr size_t guided_smem() {
    return (sizeof(TopkShared<NT>) + 15) / 16 * 16 + sizeof(GuidedShared<kCap, kBits>) + 16;
}

template <int NT, int U, int kCap, int kBits>
__global__ void __launch_bounds__(NT)
    topk_guided_kernel(const float *__restrict__ scores, int64_t stride, int64_t n,
                       int64_t offset, int32_t ratio, int64_t r0, int R, int32_t k,
                       int32_t nseg, int32_t *__restrict__ sel) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~static_cast<uintptr_t>(15));
    TopkShared<NT> &sh = *reinterpret_cast<TopkShared<NT> *>(base);
    auto *gs = reinterpret_cast<GuidedShared<kCap, kBits> *>(
        base + (sizeof(TopkShared<NT>) + 15) / 16 * 16);
    for (int it = blockIdx.x; it < R; it += gridDim.x) {
        const int row = R - 1 - it;
        const int64_t t = offset + r0 + row;
        const int64_t L = min(n, (t + 1) / ratio);
        int32_t *out = sel + (r0 + row) * static_cast<int64_t>(k);
        if (L <= k) {
            for (int i = threadIdx.x; i < k; i += NT) out[i] = i < L ? i : -1;
        } else {
            topk_row_vec<NT, U>(scores + static_cast<int64_t>(row) * stride, L, k, nseg, out, sh,
                                threadIdx.x, CtaSync{}, gs);
        }
        __syncthreads();  // the shared arrays are reused by the next row
    }
}

// Rows of up to 262,144 scores (1M tokens at ratio 4), 4096 candidates: 512-thread
// CTAs, two per SM. (For rows of up to 64K scores, which stay in L2 across the
// passes, the one-row-per-CTA kernel measured faster: 1.77 against 1.84-2.01 ms
// for score + top-k at 128K context.)
constexpr int kGuidedCap = 4096;
constexpr int kLongBits = 262144;
#define DSA_GUIDED_LONG topk_guided_kernel<kTopkThreadsLong, 4, kGuidedCap, kLongBits>
constexpr size_t kGuidedLongSmem = guided_smem<kTopkThreadsLong, 4, kGuidedCap, kLongBits>();

// Selection without scoring: sel[i, c] = c if c < n_vis(t) else -1 (n = 0: all -1).
// One CTA per row; 16-byte stores of four entries when k is a multiple of 4.
__global__ void __launch_bounds__(256) fill_selection_kernel(int32_t *sel, int32_t k,
                                                             int64_t offset, int64_t n,
                                                             int32_t ratio) {
    const int64_t i = blockIdx.x;
    const int64_t nv = min(n, (offset + i + 1) / ratio);
    int32_t *row = sel + i * k;
    if ((k & 3) == 0) {
        int4 *row4 = reinterpret_cast<int4 *>(row);
        for (int c4 = threadIdx.x; c4 < (k >> 2); c4 += blockDim.x) {
            const int c = 4 * c4;
            row4[c4] = make_int4(c < nv ? c : -1, c + 1 < nv ? c + 1 : -1,
                                 c + 2 < nv ? c + 2 : -1, c + 3 < nv ? c + 3 : -1);
        }
    } else {
        for (int c = threadIdx.x; c < k; c += blockDim.x) row[c] = c < nv ? c : -1;
    }
}

int choose_segments(int groups, int NB, int sms) {
    int best = 1;
    double best_cost = 1e30;
    // (up to 32 segments; more when the row groups alone leave SMs idle). A unit costs
    // its key blocks plus about two blocks' time of start-up (its queries' load); with 4
    // the 4096-row 128K tile took two segments per row group (7 waves of 1,024 units, the
    // last one 74 % full), with 2 it takes five (17 waves, 99 % full): score + top-k 1.502
    // against 1.535 ms, the 1M tiles unchanged
    const int cap = std::min(NB, std::max(32, sms / std::max(1, groups)));
    for (int ns = 1; ns <= cap; ++ns) {
        const int64_t units = static_cast<int64_t>(groups) * ns;
        const int64_t waves = (units + sms - 1) / sms;
        const double cost = static_cast<double>(waves) * (static_cast<double>(NB) / ns + 2.0);
        if (cost < best_cost * 0.999) {
            best_cost = cost;
            best = ns;
        }
    }
    return best;
}

}  // namespace

int launch_fill_selection(int32_t *sel, int64_t rows, int32_t k, int64_t offset, int64_t n,
                          int32_t ratio, cudaStream_t s) {
    const int threads = k >= 1024 ? 256 : (k >= 256 ? 128 : 64);
    fill_selection_kernel<<<static_cast<unsigned>(rows), threads, 0, s>>>(sel, k, offset, n,
                                                                           ratio);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// Scores of tile rows [r0, r0 + R) into `scores`.
int launch_score_tile(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const float *w, int64_t n,
                      int64_t offset, int32_t ratio, int64_t r0, int64_t R, float *scores,
                      int64_t stride, int32_t *sel, int32_t k, int *nseg_rng, int32_t *status,
                      cudaStream_t s) {
    const int sms = std::max(1, sm_count());
    ScoreParams p;
    p.w = w;
    p.scores = scores;
    p.stride = stride;
    p.n = n;
    p.offset = offset;
    p.ratio = ratio;
    p.r0 = r0;
    p.R = static_cast<int>(R);
    p.NB = static_cast<int>(stride / kScoreBlock);
    const int groups = static_cast<int>((R + kTok - 1) / kTok);
    p.nseg = choose_segments(groups, p.NB, sms);
    p.n_units = groups * p.nseg;
    // the row ranges fit the selection rows when they hold two entries per segment
    const bool rng = sel != nullptr && k >= 2 * p.nseg;
    p.rng = rng ? sel : nullptr;
    p.k = k;
    if (nseg_rng) *nseg_rng = rng ? p.nseg : 0;
    p.status = status;
    const int grid = std::min(p.n_units, sms);
    score_kernel<<<grid, kScoreThreads, kScoreSmem, s>>>(tm_q, tm_k, p);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int launch_topk_tile(const float *scores, int64_t stride, int64_t n, int64_t offset,
                     int32_t ratio, int64_t r0, int64_t R, int32_t k, int32_t nseg_rng,
                     int32_t *sel, int32_t *status, cudaStream_t s) {
    (void)status;
    const int sms = std::max(1, sm_count());
    if (n > 65536) {
        // rows over 64K scores (256 KB): two persistent 512-thread CTAs per SM with
        // 16-byte loads (a sweep at 1M context: 2 x 512 beat 1 x 1024 per SM, and both
        // beat fewer CTAs that would keep fewer rows in flight; the kernel is bound by
        // each SM's loads in flight, not by HBM). Rows up to kLongBits scores take the
        // sample-guided pass, which usually needs one pass over the row, not three.
        const int grid = static_cast<int>(std::min<int64_t>(R, 2 * sms));
        if (n <= kLongBits)
            DSA_GUIDED_LONG<<<grid, kTopkThreadsLong, kGuidedLongSmem, s>>>(
                scores, stride, n, offset, ratio, r0, static_cast<int>(R), k, nseg_rng, sel);
        else
            topk_vec_kernel<kTopkThreadsLong, 4><<<grid, kTopkThreadsLong, 0, s>>>(
                scores, stride, n, offset, ratio, r0, static_cast<int>(R), k, nseg_rng, sel);
    } else if (R < 2 * static_cast<int64_t>(sms)) {
        // few rows (decode steps, short bands): 1024-thread CTAs walk each row faster
        if (n >= kBitmapRows)
            topk_kernel<kTopkThreadsFew, true><<<static_cast<unsigned>(R), kTopkThreadsFew, 0, s>>>(
                scores, stride, n, offset, ratio, r0, k, nseg_rng, sel);
        else
            topk_kernel<kTopkThreadsFew, false><<<static_cast<unsigned>(R), kTopkThreadsFew, 0, s>>>(
                scores, stride, n, offset, ratio, r0, k, nseg_rng, sel);
    } else if (n >= kBitmapRows) {
        topk_kernel<kTopkThreads, true><<<static_cast<unsigned>(R), kTopkThreads, 0, s>>>(
            scores, stride, n, offset, ratio, r0, k, nseg_rng, sel);
    } else {
        topk_kernel<kTopkThreads, false><<<static_cast<unsigned>(R), kTopkThreads, 0, s>>>(
            scores, stride, n, offset, ratio, r0, k, nseg_rng, sel);
    }
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// Checks shared by dsa_index_score_topk and dsa_prefill_chunk.
int check_score_topk(const void *q_idx, const float *w, const void *pooled_ik, int64_t n,
                     int64_t chunk, int64_t offset, int32_t ratio, int32_t k, int64_t tile_rows,
                     const void *scratch, size_t scratch_bytes, const int32_t *sel) {
    if (!sel || chunk <= 0 || offset < 0 || n < 0) return DSA_ERR_ARG;
    if (!valid_ratio(ratio) || k <= 0 || tile_rows <= 0) return DSA_ERR_SHAPE;
    if (n != (offset + chunk) / ratio) return DSA_ERR_ARG;
    if (!aligned16(sel)) return DSA_ERR_ARG;
    if (n > k) {
        if (!q_idx || !w || !pooled_ik || !aligned16(q_idx) || !aligned16(w) ||
            !aligned16(pooled_ik))
            return DSA_ERR_ARG;
        const size_t need = dsa_score_scratch_bytes(std::min(tile_rows, chunk), n);
        if (!scratch || !aligned16(scratch) || scratch_bytes < need) return DSA_ERR_SCRATCH;
        if (chunk * kHI > (int64_t{1} << 31) - 1 || n > (int64_t{1} << 31) - 1)
            return DSA_ERR_SHAPE;
    }
    return DSA_OK;
}

namespace {

// Per-device one-time set-up of the raised shared-memory limits (score kernel,
// sample-guided top-k).
std::mutex g_score_mu;
int g_score_setup[kMaxDevices];  // 0 = not yet, else DSA_OK + 1 or the error

int score_setup() {
    const int dev = current_device();
    if (dev < 0) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_score_mu);
    if (g_score_setup[dev] == 0) {
        const bool ok =
            cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kScoreSmem) == cudaSuccess &&
            cudaFuncSetAttribute(DSA_GUIDED_LONG, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kGuidedLongSmem)) == cudaSuccess;
        g_score_setup[dev] = ok ? DSA_OK + 1 : DSA_ERR_CUDA;
    }
    return g_score_setup[dev] == DSA_OK + 1 ? DSA_OK : g_score_setup[dev];
}

}  // namespace

int prepare_score_topk(const void *q_idx, const void *pooled_ik, int64_t n, int64_t chunk,
                       int32_t k, ScoreTopkPlan *plan) {
    plan->full = n > 0 && n > k;
    if (!plan->full) return DSA_OK;
    int rc = score_setup();
    if (rc != DSA_OK) return rc;
    if (!make_tmap_bf16(&plan->tm_q, q_idx, kDI, static_cast<uint64_t>(chunk) * kHI, kDI * 2,
                        64, 256))
        return DSA_ERR_CUDA;
    if (!make_tmap_bf16(&plan->tm_k, pooled_ik, kDI, static_cast<uint64_t>(n), kDI * 2, 64, 128))
        return DSA_ERR_CUDA;
    return DSA_OK;
}

int enqueue_score_topk(const ScoreTopkPlan &plan, const float *w, int64_t n, int64_t offset,
                       int32_t ratio, int32_t k, int64_t r_begin, int64_t r_end,
                       int64_t tile_rows, void *scratch, int32_t *sel, int32_t *status,
                       cudaStream_t s) {
    if (r_end <= r_begin) return DSA_OK;
    if (!plan.full)
        return launch_fill_selection(sel + r_begin * k, r_end - r_begin, k, offset + r_begin, n,
                                     ratio, s);
    const int64_t stride = score_stride(n);
    float *scores = static_cast<float *>(scratch);
    for (int64_t r0 = r_begin; r0 < r_end; r0 += tile_rows) {
        const int64_t R = std::min(tile_rows, r_end - r0);
        int nseg_rng = 0;
        int rc = launch_score_tile(plan.tm_q, plan.tm_k, w, n, offset, ratio, r0, R, scores,
                                   stride, sel, k, &nseg_rng, status, s);
        if (rc != DSA_OK) return rc;
        rc = launch_topk_tile(scores, stride, n, offset, ratio, r0, R, k, nseg_rng, sel, status, s);
        if (rc != DSA_OK) return rc;
    }
    return DSA_OK;
}

}  // namespace dsa

extern "C" size_t dsa_score_scratch_bytes(int64_t tile_rows, int64_t n_pooled) {
    if (tile_rows <= 0 || n_pooled <= 0) return 0;
    return static_cast<size_t>(tile_rows) * static_cast<size_t>(dsa::score_stride(n_pooled)) *
           sizeof(float);
}

extern "C" int dsa_index_score_topk(const void *q_idx, const float *w, const void *pooled_ik,
                                    int64_t n_pooled, int64_t chunk, int64_t offset, int32_t ratio,
                                    int32_t index_topk, int64_t tile_rows, void *scratch,
                                    size_t scratch_bytes, int32_t *sel, int32_t *dev_status,
                                    void *stream) {
    using namespace dsa;
    int rc = check_score_topk(q_idx, w, pooled_ik, n_pooled, chunk, offset, ratio, index_topk,
                              tile_rows, scratch, scratch_bytes, sel);
    if (rc != DSA_OK) return rc;
    ScoreTopkPlan plan;
    rc = prepare_score_topk(q_idx, pooled_ik, n_pooled, chunk, index_topk, &plan);
    if (rc != DSA_OK) return rc;
    return enqueue_score_topk(plan, w, n_pooled, offset, ratio, index_topk, 0, chunk, tile_rows,
                              scratch, sel, dev_status, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ no-allocation variant
//
// Score scratch held by the library itself, for callers that cannot hand it
// device memory. Every device that loads the library keeps this array until
// the process exits; all calls on a device share it.
namespace dsa {
namespace {

__device__ __align__(256) static float g_static_scratch[DSA_STATIC_SCRATCH_BYTES / sizeof(float)];

// The current context's unique id, 0 when there is none yet or it cannot be read.
// A device reset destroys the context together with the module that holds the
// array, so a cached address is reused only while the id stays the same.
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

struct StaticScratch {
    unsigned long long ctx_id = 0;
    void *ptr = nullptr;
};
std::mutex g_static_mu;
StaticScratch g_static[kMaxDevices];

// Device address of g_static_scratch on the current device (the host-side name
// of the array is only a stand-in, not a device address). Looked up on the first
// call on a device, and again only if the device's context has changed since.
int static_scratch(void **out) {
    const int dev = current_device();
    if (dev < 0) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_static_mu);
    StaticScratch &c = g_static[dev];
    const unsigned long long id = current_context_id();
    if (!c.ptr || id == 0 || id != c.ctx_id) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr)
            return DSA_ERR_CUDA;
        c.ptr = ptr;
        c.ctx_id = current_context_id();
    }
    *out = c.ptr;
    return DSA_OK;
}

}  // namespace
}  // namespace dsa

extern "C" int dsa_index_score_topk_noalloc(const void *q_idx, const float *w,
                                            const void *pooled_ik, int64_t n_pooled,
                                            int64_t chunk, int64_t offset, int32_t ratio,
                                            int32_t index_topk, int64_t tile_rows, int32_t *sel,
                                            int32_t *dev_status, void *stream) {
    using namespace dsa;
    // validate with the library-held scratch standing in for the caller's buffer
    const void *probe = reinterpret_cast<const void *>(uintptr_t{256});
    int rc = check_score_topk(q_idx, w, pooled_ik, n_pooled, chunk, offset, ratio, index_topk,
                              tile_rows, probe, DSA_STATIC_SCRATCH_BYTES, sel);
    if (rc != DSA_OK) return rc;
    void *scratch = nullptr;
    if (n_pooled > index_topk) {
        rc = static_scratch(&scratch);
        if (rc != DSA_OK) return rc;
    }
    ScoreTopkPlan plan;
    rc = prepare_score_topk(q_idx, pooled_ik, n_pooled, chunk, index_topk, &plan);
    if (rc != DSA_OK) return rc;
    return enqueue_score_topk(plan, w, n_pooled, offset, ratio, index_topk, 0, chunk, tile_rows,
                              scratch, sel, dev_status, static_cast<cudaStream_t>(stream));
}
