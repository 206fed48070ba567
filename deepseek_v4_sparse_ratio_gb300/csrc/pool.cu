// Step (a): mean pooling of a chunk's raw rows into the PoolingCache (ratio 4
// for the indexed attention; any power of two up to 128, e.g. the compressed
// attention's 128).
//
// "perf(deepseek-v4): skip redundant all-pooled indexer scoring", Summary and
// Correctness: the attention-KV and indexer-key compressors both run once per
// chunk, and a non-aligned chunk carries its last (tokens mod 4) raw rows to
// the next one. "perf(deepseek_v4): faster exact DeepSeek-V4 prefill",
// Summary item 4: new pooled rows are written in place after the existing
// ones, with no re-concatenation of the prefix.
//
// Arithmetic: a pooled element is the mean of `ratio` bf16 values (a power of
// two up to 128: the fp64 sum, taken in row order, is exact for such values in
// practice, and /ratio is exact), rounded once to bf16 with ties to even.
// GB300's fp64 rate is a small fraction of its fp32 rate, so the sum is first
// taken in fp32 with an error-free check of every addition (TwoSum); only when
// some fp32 partial sum rounded is it taken again in fp64. While every fp32
// partial sum is exact, the fp64 partial sums are the same values, so the
// result is the fp64 row-order sum either way.
// HBM-bound: each thread moves one 16-byte vector of each of the raw rows and
// writes one 16-byte vector of the pooled row.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace dsa {

namespace {

constexpr int kVecKV = kD * 2 / 16;   // 64 16-byte vectors per KV row
constexpr int kVecIK = kDI * 2 / 16;  // 16 per indexer-key row
constexpr int kVecRow = kVecKV + kVecIK;

// Round a double to the nearest bf16 (ties to even), straight from the
// double's bits so that no intermediate fp32 rounding happens.
__device__ __forceinline__ uint32_t bf16_rne_from_double(double x) {
    const uint64_t b = static_cast<uint64_t>(__double_as_longlong(x));
    const uint32_t sign = static_cast<uint32_t>(b >> 48) & 0x8000u;
    const uint64_t mag = b & 0x7FFFFFFFFFFFFFFFull;
    if (mag > 0x7FF0000000000000ull) return 0x7FC0u;
    const int e = static_cast<int>(mag >> 52) - 1023;
    if (e >= 128) return sign | 0x7F80u;
    if (e < -126) {
        // below the smallest normal: the bf16 grid spacing is 2^-133
        const double sc = __longlong_as_double(static_cast<long long>(mag)) * 0x1p133;
        return sign | static_cast<uint32_t>(rint(sc));
    }
    uint64_t v = (static_cast<uint64_t>(e + 127) << 52) | (mag & ((1ull << 52) - 1));
    v += ((1ull << 44) - 1) + ((v >> 45) & 1ull);  // round the 45 dropped bits, ties to even
    const uint32_t r = static_cast<uint32_t>(v >> 45);
    return sign | (r >= 0x7F80u ? 0x7F80u : r);
}

// a + b rounded to fp32; sets `bit` in `inexact` when that rounding lost
// anything (Knuth's TwoSum: s + err == a + b exactly; an infinity or NaN gives
// err NaN).
__device__ __forceinline__ float add_checked(float a, float b, uint32_t &inexact, uint32_t bit) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    if (!(err == 0.0f)) inexact |= bit;
    return s;
}

__device__ __forceinline__ void add8_checked(float (&acc)[8], uint4 x, uint32_t &inexact) {
    acc[0] = add_checked(acc[0], bf16lo(x.x), inexact, 1u);
    acc[1] = add_checked(acc[1], bf16hi(x.x), inexact, 2u);
    acc[2] = add_checked(acc[2], bf16lo(x.y), inexact, 4u);
    acc[3] = add_checked(acc[3], bf16hi(x.y), inexact, 8u);
    acc[4] = add_checked(acc[4], bf16lo(x.z), inexact, 16u);
    acc[5] = add_checked(acc[5], bf16hi(x.z), inexact, 32u);
    acc[6] = add_checked(acc[6], bf16lo(x.w), inexact, 64u);
    acc[7] = add_checked(acc[7], bf16hi(x.w), inexact, 128u);
}

// Element e (0..7) of a 16-byte vector of bf16 values.
__device__ __forceinline__ float elem8(uint4 x, int e) {
    const uint32_t w = e < 2 ? x.x : e < 4 ? x.y : e < 6 ? x.z : x.w;
    return (e & 1) ? bf16hi(w) : bf16lo(w);
}

// One thread per (new pooled row, 16-byte vector): 64 vectors of KV then 16
// of indexer keys. Raw token u = 4g+i comes from the remainder if u < offset,
// else from chunk row u - offset.
__global__ void __launch_bounds__(256) pool_kernel(const uint4 *__restrict__ raw_kv,
                                                   const uint4 *__restrict__ raw_ik,
                                                   const uint4 *__restrict__ rem_kv,
                                                   const uint4 *__restrict__ rem_ik,
                                                   uint4 *__restrict__ pooled_kv,
                                                   uint4 *__restrict__ pooled_ik, int64_t n_old,
                                                   int64_t n_new, int64_t offset, int32_t ratio) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= (n_new - n_old) * kVecRow) return;
    const int64_t g = n_old + idx / kVecRow;
    const int v = static_cast<int>(idx % kVecRow);
    const bool is_kv = v < kVecKV;
    const int vv = is_kv ? v : v - kVecKV;
    const int per_row = is_kv ? kVecKV : kVecIK;
    const uint4 *raw = is_kv ? raw_kv : raw_ik;
    const uint4 *rem = is_kv ? rem_kv : rem_ik;
    const int64_t rem_base = n_old * ratio;  // absolute token held in remainder slot 0

    auto row = [&](int i) {
        const int64_t u = g * ratio + i;
        return (u < offset) ? rem[(u - rem_base) * per_row + vv]
                            : __ldg(&raw[(u - offset) * per_row + vv]);
    };
    // rows are loaded kBatch at a time, all in flight before any is summed
    constexpr int kBatch = 8;
    float acc32[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    uint32_t inexact = 0;  // bit e: element e's fp32 running sum rounded somewhere
    for (int i0 = 0; i0 < ratio; i0 += kBatch) {
        uint4 x[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (i0 + j < ratio) x[j] = row(i0 + j);
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (i0 + j < ratio) add8_checked(acc32, x[j], inexact);
    }
    double acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = acc32[e];
    // only the elements whose fp32 sum rounded are summed again, in fp64
    while (inexact) {
        const int e = __ffs(inexact) - 1;
        inexact &= inexact - 1;
        double a = 0.0;
        for (int i0 = 0; i0 < ratio; i0 += kBatch) {
            float y[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (i0 + j < ratio) y[j] = elem8(row(i0 + j), e);
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (i0 + j < ratio) a += y[j];
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k == e) acc[k] = a;  // (a static index keeps acc in registers)
    }
    uint32_t o[8];
    const double inv = 1.0 / ratio;  // exact: ratio is a power of two
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = bf16_rne_from_double(acc[e] * inv);
    uint4 out;
    out.x = o[0] | (o[1] << 16);
    out.y = o[2] | (o[3] << 16);
    out.z = o[4] | (o[5] << 16);
    out.w = o[6] | (o[7] << 16);
    (is_kv ? pooled_kv : pooled_ik)[g * per_row + vv] = out;
}

constexpr int kWordKV = kD / 2;   // 256 4-byte words (bf16 pairs) per KV row
constexpr int kWordIK = kDI / 2;  // 64 per indexer-key row
constexpr int kWordRow = kWordKV + kWordIK;

// The same mean for large ratios: one thread per (new pooled row, 4-byte
// word), so that a thread keeps 32 raw rows in flight rather than 8 (with
// `ratio` rows to sum, a thread is bound by its chain of loads).
__global__ void __launch_bounds__(256) pool_words_kernel(const uint32_t *__restrict__ raw_kv,
                                                         const uint32_t *__restrict__ raw_ik,
                                                         const uint32_t *__restrict__ rem_kv,
                                                         const uint32_t *__restrict__ rem_ik,
                                                         uint32_t *__restrict__ pooled_kv,
                                                         uint32_t *__restrict__ pooled_ik,
                                                         int64_t n_old, int64_t n_new,
                                                         int64_t offset, int32_t ratio) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= (n_new - n_old) * kWordRow) return;
    const int64_t g = n_old + idx / kWordRow;
    const int v = static_cast<int>(idx % kWordRow);
    const bool is_kv = v < kWordKV;
    const int vv = is_kv ? v : v - kWordKV;
    const int per_row = is_kv ? kWordKV : kWordIK;
    const uint32_t *raw = is_kv ? raw_kv : raw_ik;
    const uint32_t *rem = is_kv ? rem_kv : rem_ik;
    // row i of the group: remainder slot or chunk row (one pointer step per row)
    const int64_t u0 = g * ratio;
    const uint32_t *rem_p = rem + (u0 - n_old * ratio) * per_row + vv;
    const uint32_t *raw_p = raw + (u0 - offset) * per_row + vv;
    auto row = [&](int i) {
        return (u0 + i < offset) ? rem_p[i * per_row] : __ldg(raw_p + i * per_row);
    };
    constexpr int kBatch = 32;
    float a0 = 0.0f, a1 = 0.0f;
    uint32_t inexact = 0;
    for (int i0 = 0; i0 < ratio; i0 += kBatch) {
        uint32_t x[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (i0 + j < ratio) x[j] = row(i0 + j);
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (i0 + j < ratio) {
                a0 = add_checked(a0, bf16lo(x[j]), inexact, 1u);
                a1 = add_checked(a1, bf16hi(x[j]), inexact, 2u);
            }
    }
    double d0 = a0, d1 = a1;
    if (inexact) {
        // some fp32 partial sum rounded: both sums again in fp64, in row order
        d0 = 0.0;
        d1 = 0.0;
        for (int i0 = 0; i0 < ratio; i0 += kBatch) {
            uint32_t x[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (i0 + j < ratio) x[j] = row(i0 + j);
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (i0 + j < ratio) {
                    d0 += bf16lo(x[j]);
                    d1 += bf16hi(x[j]);
                }
        }
    }
    const double inv = 1.0 / ratio;  // exact: ratio is a power of two
    (is_kv ? pooled_kv : pooled_ik)[g * per_row + vv] =
        bf16_rne_from_double(d0 * inv) | (bf16_rne_from_double(d1 * inv) << 16);
}

// Copy the chunk rows that form the new remainder (tokens 4*n_new .. end-1
// that come from this chunk) into their remainder slots. Remainder tokens
// that predate the chunk already sit in their slot.
__global__ void remainder_kernel(const uint4 *__restrict__ raw_kv, const uint4 *__restrict__ raw_ik,
                                 uint4 *__restrict__ rem_kv, uint4 *__restrict__ rem_ik,
                                 int64_t n_new, int64_t offset, int64_t end, int32_t ratio) {
    const int64_t first = n_new * ratio > offset ? n_new * ratio : offset;
    const int64_t rows = end - first;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
         idx < rows * kVecRow; idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t u = first + idx / kVecRow;
        const int v = static_cast<int>(idx % kVecRow);
        const int64_t slot = u - n_new * ratio;
        if (v < kVecKV)
            rem_kv[slot * kVecKV + v] = raw_kv[(u - offset) * kVecKV + v];
        else
            rem_ik[slot * kVecIK + (v - kVecKV)] = raw_ik[(u - offset) * kVecIK + (v - kVecKV)];
    }
}

}  // namespace

int launch_pool_append(const dsa_pool_state &st, const void *raw_kv, const void *raw_ik,
                       int64_t chunk, int64_t offset, cudaStream_t s) {
    const int64_t n_old = st.n_pooled_kv;
    const int32_t ratio = st.ratio;
    const int64_t end = offset + chunk;
    const int64_t n_new = end / ratio;
    if (n_new > n_old) {
        // large ratios: a thread per 4-byte word; few new rows: smaller blocks
        // spread them over more SMs
        const bool words = ratio >= 32;
        const int64_t threads = (n_new - n_old) * (words ? kWordRow : kVecRow);
        const int bs = (threads + 255) / 256 >= 2 * static_cast<int64_t>(sm_count()) ? 256 : 64;
        const int64_t blocks = (threads + bs - 1) / bs;
        if (words)
            pool_words_kernel<<<static_cast<unsigned>(blocks), bs, 0, s>>>(
                static_cast<const uint32_t *>(raw_kv), static_cast<const uint32_t *>(raw_ik),
                static_cast<const uint32_t *>(st.rem_kv), static_cast<const uint32_t *>(st.rem_ik),
                static_cast<uint32_t *>(st.pooled_kv), static_cast<uint32_t *>(st.pooled_ik),
                n_old, n_new, offset, ratio);
        else
            pool_kernel<<<static_cast<unsigned>(blocks), bs, 0, s>>>(
                static_cast<const uint4 *>(raw_kv), static_cast<const uint4 *>(raw_ik),
                static_cast<const uint4 *>(st.rem_kv), static_cast<const uint4 *>(st.rem_ik),
                static_cast<uint4 *>(st.pooled_kv), static_cast<uint4 *>(st.pooled_ik), n_old,
                n_new, offset, ratio);
        if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
    }
    if (end % ratio != 0) {
        const int64_t threads = (end % ratio) * kVecRow;
        remainder_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(
            static_cast<const uint4 *>(raw_kv), static_cast<const uint4 *>(raw_ik),
            static_cast<uint4 *>(st.rem_kv), static_cast<uint4 *>(st.rem_ik), n_new, offset, end,
            ratio);
        if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

// ------------------------------------------------------------------ host helpers

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

bool make_tmap_bf16(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, bool swizzle128) {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace dsa

// ------------------------------------------------------------------ C ABI

extern "C" int dsa_pool_append(dsa_pool_state *st, const void *raw_kv, const void *raw_ik,
                               int64_t chunk, int64_t offset, int32_t ratio, void *stream) {
    using namespace dsa;
    if (!st || !raw_kv || !raw_ik || chunk <= 0 || offset < 0) return DSA_ERR_ARG;
    if (!st->pooled_kv || !st->pooled_ik || !st->rem_kv || !st->rem_ik) return DSA_ERR_ARG;
    if (!aligned16(raw_kv) || !aligned16(raw_ik) || !aligned16(st->pooled_kv) ||
        !aligned16(st->pooled_ik) || !aligned16(st->rem_kv) || !aligned16(st->rem_ik))
        return DSA_ERR_ARG;
    if (!valid_ratio(ratio) || st->ratio != ratio) return DSA_ERR_SHAPE;
    if (st->n_pooled_kv != st->n_pooled_ik) return DSA_ERR_DIVERGED;
    if (st->n_rem < 0 || st->n_rem >= ratio || st->n_pooled_kv < 0 ||
        st->n_pooled_kv * ratio + st->n_rem != st->n_tokens)
        return DSA_ERR_ARG;
    if (offset != st->n_tokens) return DSA_ERR_OFFSET;
    const int64_t end = offset + chunk;
    const int64_t n_new = end / ratio;
    if (n_new > st->cap) return DSA_ERR_CAPACITY;
    int rc = launch_pool_append(*st, raw_kv, raw_ik, chunk, offset,
                                static_cast<cudaStream_t>(stream));
    if (rc != DSA_OK) return rc;
    st->n_pooled_kv = st->n_pooled_ik = n_new;
    st->n_tokens = end;
    st->n_rem = static_cast<int32_t>(end % ratio);
    return DSA_OK;
}

extern "C" const char *dsa_strerror(int code) {
    switch (code) {
        case DSA_OK: return "ok";
        case DSA_ERR_ARG: return "invalid argument (null, non-positive size or misaligned pointer)";
        case DSA_ERR_SHAPE:
            return "unsupported shape (ratio not a power of two in [2,128], index_topk, window or tile)";
        case DSA_ERR_OFFSET: return "chunk offset does not match the tokens already in the cache";
        case DSA_ERR_CAPACITY: return "pooled cache capacity exceeded";
        case DSA_ERR_DIVERGED: return "attention and indexer pooled caches hold different row counts";
        case DSA_ERR_SCRATCH: return "score scratch missing or too small";
        case DSA_ERR_CUDA: return "CUDA launch or driver call failed";
        case DSA_ERR_TIMEOUT: return "a bounded wait inside a kernel expired";
        case DSA_ERR_BOUNDS: return "an index was outside its buffer (access skipped)";
        case DSA_ERR_RAW_RANGE: return "raw KV buffer does not cover the window and the chunk";
        default: return "unknown status";
    }
}
