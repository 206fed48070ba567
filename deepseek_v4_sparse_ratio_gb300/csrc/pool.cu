// Step (a): ratio-4 mean pooling of a chunk's raw rows into the PoolingCache.
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

__device__ __forceinline__ void add8(double (&acc)[8], uint4 x) {
    acc[0] += bf16lo(x.x); acc[1] += bf16hi(x.x);
    acc[2] += bf16lo(x.y); acc[3] += bf16hi(x.y);
    acc[4] += bf16lo(x.z); acc[5] += bf16hi(x.z);
    acc[6] += bf16lo(x.w); acc[7] += bf16hi(x.w);
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

    double acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll 4
    for (int i = 0; i < ratio; ++i) {
        const int64_t u = g * ratio + i;
        const uint4 x = (u < offset) ? rem[(u - rem_base) * per_row + vv]
                                     : __ldg(&raw[(u - offset) * per_row + vv]);
        add8(acc, x);
    }
    uint32_t o[8];
#pragma unroll
    const double inv = 1.0 / ratio;  // exact: ratio is a power of two
    for (int e = 0; e < 8; ++e) o[e] = bf16_rne_from_double(acc[e] * inv);
    uint4 out;
    out.x = o[0] | (o[1] << 16);
    out.y = o[2] | (o[3] << 16);
    out.z = o[4] | (o[5] << 16);
    out.w = o[6] | (o[7] << 16);
    (is_kv ? pooled_kv : pooled_ik)[g * per_row + vv] = out;
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
        const int64_t threads = (n_new - n_old) * kVecRow;
        const int64_t blocks = (threads + 255) / 256;
        pool_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
            static_cast<const uint4 *>(raw_kv), static_cast<const uint4 *>(raw_ik),
            static_cast<const uint4 *>(st.rem_kv), static_cast<const uint4 *>(st.rem_ik),
            static_cast<uint4 *>(st.pooled_kv), static_cast<uint4 *>(st.pooled_ik), n_old, n_new,
            offset, ratio);
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
