// Host-side internals shared by the translation units of libdsa.so: launch
// entry points of each kernel family, tensor-map construction and argument checks.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

constexpr int kRatio = DSA_RATIO;
constexpr int kHI = DSA_INDEX_HEADS;
constexpr int kDI = DSA_INDEX_DIM;
constexpr int kH = DSA_HEADS;
constexpr int kD = DSA_DIM;

// Pooled rows per score block (MMA M), and the padded row stride of the score
// scratch in floats.
constexpr int kScoreBlock = 128;
inline int64_t score_stride(int64_t n_pooled) {
    return (n_pooled + kScoreBlock - 1) / kScoreBlock * kScoreBlock;
}

// Pooling ratios the library accepts: powers of two in [2, 128] (4 for the
// indexed attention, 128 for the compressed attention).
constexpr int kMaxRatio = 128;
inline bool valid_ratio(int64_t r) { return r >= 2 && r <= kMaxRatio && (r & (r - 1)) == 0; }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D bf16 tensor map: `inner` elements per row (the contiguous dimension),
// `rows` rows of `row_bytes` each, box of box_inner x box_rows, 128-byte
// swizzle or none. Returns false if the driver rejects it.
bool make_tmap_bf16(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                    bool swizzle128 = true);

int sm_count();

// Launchers (stream-ordered, no host synchronization). Each returns DSA_OK or
// DSA_ERR_CUDA; arguments are validated by the caller.
int launch_pool_append(const dsa_pool_state &st, const void *raw_kv, const void *raw_ik,
                       int64_t chunk, int64_t offset, cudaStream_t s);
int launch_fill_selection(int32_t *sel, int64_t rows, int32_t k, int64_t offset, int64_t n,
                          int32_t ratio, cudaStream_t s);
// launch_score_tile also writes each row's per-segment score range into the
// row's selection entries when k >= 2 x segments (sel may be null) and reports
// the segment count in *nseg_rng (0 when it did not); launch_topk_tile then
// takes the range from there (nseg_rng > 0) instead of a pass over the scores.
int launch_score_tile(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const float *w,
                      int64_t n, int64_t offset, int32_t ratio, int64_t r0, int64_t R,
                      float *scores, int64_t stride, int32_t *sel, int32_t k, int *nseg_rng,
                      int32_t *status, cudaStream_t s);
int launch_topk_tile(const float *scores, int64_t stride, int64_t n, int64_t offset,
                     int32_t ratio, int64_t r0, int64_t R, int32_t k, int32_t nseg_rng,
                     int32_t *sel, int32_t *status, cudaStream_t s);
int launch_attention(const void *q, const void *raw_kv, int64_t raw_start, int64_t raw_rows,
                     const void *pooled_kv, int64_t n, const int32_t *sel, int32_t k,
                     int64_t chunk, int64_t offset, int32_t ratio, int32_t window, float scale,
                     void *out, int32_t *status, cudaStream_t s);

}  // namespace dsa
