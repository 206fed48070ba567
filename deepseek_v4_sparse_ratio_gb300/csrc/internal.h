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

// One-time set-up (raised shared-memory limits, occupancy probes) is per device:
// each launcher keeps it in a table indexed by the current device's ordinal.
constexpr int kMaxDevices = 64;
int current_device();  // the current device's ordinal, or -1 when unusable

// Each step is split in two: prepare_* does everything that can fail short of a
// launch (argument-derived tensor maps, per-device set-up) and enqueue_* only
// launches. The whole-chunk calls prepare every step before enqueuing any, so a
// rejected call enqueues nothing.

// Launchers (stream-ordered, no host synchronization). Each returns DSA_OK or
// DSA_ERR_CUDA; arguments are validated by the caller.
int launch_pool_append(const dsa_pool_state &st, const void *raw_kv, const void *raw_ik,
                       int64_t chunk, int64_t offset, cudaStream_t s);
int launch_fill_selection(int32_t *sel, int64_t rows, int32_t k, int64_t offset, int64_t n,
                          int32_t ratio, cudaStream_t s);

// Score + top-k of one chunk (steps b, c): the full path when n > k.
struct ScoreTopkPlan {
    bool full = false;
    CUtensorMap tm_q, tm_k;
};
int check_score_topk(const void *q_idx, const float *w, const void *pooled_ik, int64_t n,
                     int64_t chunk, int64_t offset, int32_t ratio, int32_t k, int64_t tile_rows,
                     const void *scratch, size_t scratch_bytes, const int32_t *sel);
int prepare_score_topk(const void *q_idx, const void *pooled_ik, int64_t n, int64_t chunk,
                       int32_t k, ScoreTopkPlan *plan);
// Rows [r_begin, r_end) of the chunk, in tiles of at most tile_rows rows (each tile's
// scores start at the scratch's first row); `plan` covers the whole chunk.
int enqueue_score_topk(const ScoreTopkPlan &plan, const float *w, int64_t n, int64_t offset,
                       int32_t ratio, int32_t k, int64_t r_begin, int64_t r_end,
                       int64_t tile_rows, void *scratch, int32_t *sel, int32_t *status,
                       cudaStream_t s);

// Window + selected attention (step d).
struct AttnPlan {
    CUtensorMap tm_q;
    bool split_ok = false;  // the cluster launch of the split mode can be resident
};
int check_attention(const void *q, const void *raw_kv, int64_t raw_start, int64_t raw_rows,
                    const void *pooled_kv, int64_t n, const int32_t *sel, int32_t k,
                    int64_t chunk, int64_t offset, int32_t ratio, int32_t window, float scale,
                    const void *out);
int prepare_attention(const void *q, int64_t chunk, AttnPlan *plan);
int enqueue_attention(const AttnPlan &plan, const void *raw_kv, int64_t raw_start,
                      const void *pooled_kv, int64_t n, const int32_t *sel, int32_t k,
                      int64_t chunk, int64_t offset, int32_t ratio, int32_t window, float scale,
                      void *out, int32_t *status, cudaStream_t s);

}  // namespace dsa
