// Step (d): exact attention of each query over its raw sliding window plus
// its selected pooled rows.
//
// "perf(deepseek_v4): faster exact DeepSeek-V4 prefill", Summary item 1: one
// fused kernel for the windowed + pooled prefill attention of DeepSeek-V4
// (B=1, H=64, D=512, bf16) that rebuilds causality, the sliding window and
// pooled visibility from offsets instead of taking a mask.
// "[Discussion] Tile indexed-attention scoring independently of the global
// prefill chunk", Possible design step 4: the selected rows feed the indexed
// attention.
//
// Keys of (t, h): raw rows u = max(0, t-W+1) .. t, then pooled rows sel[t, :]
// that are >= 0. One 512-wide row is both key and value for all 64 heads.
// Softmax runs online in fp32 (exp2 of log2e-scaled logits); the output is
// normalised once at the end and stored as bf16.
//
// This version is one warp per (token, head): lane l owns dims 16l..16l+15 of
// q, of every key row it reads, and of the output accumulator.
#include <math.h>

#include "common.cuh"

namespace dsa {

namespace {

constexpr int kAttnWarps = 8;  // heads per CTA

__device__ __forceinline__ void load16(const __nv_bfloat16 *p, float (&x)[16]) {
    const uint4 *v = reinterpret_cast<const uint4 *>(p);
    const uint4 a = __ldg(v), b = __ldg(v + 1);
    x[0] = bf16lo(a.x); x[1] = bf16hi(a.x); x[2] = bf16lo(a.y); x[3] = bf16hi(a.y);
    x[4] = bf16lo(a.z); x[5] = bf16hi(a.z); x[6] = bf16lo(a.w); x[7] = bf16hi(a.w);
    x[8] = bf16lo(b.x); x[9] = bf16hi(b.x); x[10] = bf16lo(b.y); x[11] = bf16hi(b.y);
    x[12] = bf16lo(b.z); x[13] = bf16hi(b.z); x[14] = bf16lo(b.w); x[15] = bf16hi(b.w);
}

struct AttnParams {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *raw_kv;
    int64_t raw_start;
    const __nv_bfloat16 *pooled_kv;
    int64_t n;
    const int32_t *sel;
    int32_t k;
    int64_t offset;
    int32_t window;
    float scale_log2;  // softmax scale * log2(e)
    __nv_bfloat16 *out;
    int32_t *status;
};

__device__ __forceinline__ void attend_row(const __nv_bfloat16 *row, int lane, const float (&qv)[16],
                                           float scale_log2, float &m, float &l, float (&o)[16]) {
    float kv[16];
    load16(row + lane * 16, kv);
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s = fmaf(qv[i], kv[i], s);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
    s *= scale_log2;
    const float m_new = fmaxf(m, s);
    const float corr = exp2f(m - m_new);
    const float pr = exp2f(s - m_new);
    l = l * corr + pr;
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i] = fmaf(pr, kv[i], o[i] * corr);
    m = m_new;
}

__global__ void __launch_bounds__(kAttnWarps * 32) attn_warp_kernel(const AttnParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t i = blockIdx.x / (kH / kAttnWarps);
    const int h = (blockIdx.x % (kH / kAttnWarps)) * kAttnWarps + warp;
    const int64_t t = p.offset + i;
    float qv[16];
    load16(p.q + (i * kH + h) * kD + lane * 16, qv);
    float m = -INFINITY, l = 0.0f, o[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) o[e] = 0.0f;

    const int64_t u0 = t - p.window + 1 > 0 ? t - p.window + 1 : 0;
    for (int64_t u = u0; u <= t; ++u)
        attend_row(p.raw_kv + (u - p.raw_start) * kD, lane, qv, p.scale_log2, m, l, o);
    const int64_t nv = min(p.n, (t + 1) / kRatio);
    const int32_t *srow = p.sel + i * p.k;
    for (int c = 0; c < p.k; ++c) {
        const int32_t j = __ldg(&srow[c]);
        if (j < 0) continue;
        if (j >= nv) {
            if (lane == 0 && h == 0) report(p.status, DSA_ERR_BOUNDS);
            continue;
        }
        attend_row(p.pooled_kv + static_cast<int64_t>(j) * kD, lane, qv, p.scale_log2, m, l, o);
    }
    const float inv = 1.0f / l;
    uint32_t packed[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(o[2 * e] * inv, o[2 * e + 1] * inv);
        packed[e] = *reinterpret_cast<const uint32_t *>(&v);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (i * kH + h) * kD + lane * 16);
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
}

}  // namespace

int launch_attention(const void *q, const void *raw_kv, int64_t raw_start, int64_t raw_rows,
                     const void *pooled_kv, int64_t n, const int32_t *sel, int32_t k,
                     int64_t chunk, int64_t offset, int32_t window, float scale, void *out,
                     int32_t *status, cudaStream_t s) {
    (void)raw_rows;
    AttnParams p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.raw_kv = static_cast<const __nv_bfloat16 *>(raw_kv);
    p.raw_start = raw_start;
    p.pooled_kv = static_cast<const __nv_bfloat16 *>(pooled_kv);
    p.n = n;
    p.sel = sel;
    p.k = k;
    p.offset = offset;
    p.window = window;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.status = status;
    const int64_t blocks = chunk * (kH / kAttnWarps);
    attn_warp_kernel<<<static_cast<unsigned>(blocks), kAttnWarps * 32, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int check_attention(const void *q, const void *raw_kv, int64_t raw_start, int64_t raw_rows,
                    const void *pooled_kv, int64_t n, const int32_t *sel, int32_t k,
                    int64_t chunk, int64_t offset, int32_t ratio, int32_t window, float scale,
                    const void *out) {
    if (!q || !raw_kv || !sel || !out || chunk <= 0 || offset < 0 || n < 0 || raw_rows <= 0)
        return DSA_ERR_ARG;
    if (n > 0 && !pooled_kv) return DSA_ERR_ARG;
    if (!aligned16(q) || !aligned16(raw_kv) || !aligned16(sel) || !aligned16(out) ||
        (pooled_kv && !aligned16(pooled_kv)))
        return DSA_ERR_ARG;
    if (ratio != kRatio || k <= 0 || window <= 0 || !(scale > 0.0f) || isinf(scale))
        return DSA_ERR_SHAPE;
    const int64_t first = offset - window + 1 > 0 ? offset - window + 1 : 0;
    if (raw_start > first || raw_start + raw_rows < offset + chunk) return DSA_ERR_RAW_RANGE;
    return DSA_OK;
}

}  // namespace dsa

extern "C" int dsa_window_sparse_attn(const void *q, const void *raw_kv, int64_t raw_start,
                                      int64_t raw_rows, const void *pooled_kv, int64_t n_pooled,
                                      const int32_t *sel, int32_t index_topk, int64_t chunk,
                                      int64_t offset, int32_t ratio, int32_t window, float scale,
                                      void *out, int32_t *dev_status, void *stream) {
    using namespace dsa;
    int rc = check_attention(q, raw_kv, raw_start, raw_rows, pooled_kv, n_pooled, sel, index_topk,
                             chunk, offset, ratio, window, scale, out);
    if (rc != DSA_OK) return rc;
    return launch_attention(q, raw_kv, raw_start, raw_rows, pooled_kv, n_pooled, sel, index_topk,
                            chunk, offset, window, scale, out, dev_status,
                            static_cast<cudaStream_t>(stream));
}
