// The whole path for one chunk: pool/append, score + top-k (or the skip path),
// window + selected attention, enqueued in order on one stream with every
// argument checked before the first launch.
//
// "perf(deepseek_v4): faster exact DeepSeek-V4 prefill", Summary (one prefill
// step per chunk; the compressor runs in every step) and "[Discussion] Tile
// indexed-attention scoring independently of the global prefill chunk",
// Possible design (a global chunk whose indexer work runs in bounded tiles).
#include "common.cuh"

namespace dsa {
int check_score_topk(const void *q_idx, const float *w, const void *pooled_ik, int64_t n,
                     int64_t chunk, int64_t offset, int32_t ratio, int32_t k, int64_t tile_rows,
                     const void *scratch, size_t scratch_bytes, const int32_t *sel);
int run_score_topk(const void *q_idx, const float *w, const void *pooled_ik, int64_t n,
                   int64_t chunk, int64_t offset, int32_t ratio, int32_t k, int64_t tile_rows,
                   void *scratch, int32_t *sel, int32_t *status, cudaStream_t s);
int check_attention(const void *q, const void *raw_kv, int64_t raw_start, int64_t raw_rows,
                    const void *pooled_kv, int64_t n, const int32_t *sel, int32_t k,
                    int64_t chunk, int64_t offset, int32_t ratio, int32_t window, float scale,
                    const void *out);
}  // namespace dsa

extern "C" int dsa_prefill_chunk(dsa_pool_state *st, const void *raw_kv, int64_t raw_start,
                                 int64_t raw_rows, const void *raw_ik, const void *q_idx,
                                 const float *w, const void *q, int64_t chunk, int64_t offset,
                                 int32_t index_topk, int32_t window, float scale,
                                 int64_t tile_rows, void *scratch, size_t scratch_bytes,
                                 int32_t *sel, void *out, int32_t *dev_status, void *stream) {
    using namespace dsa;
    if (!st || !raw_kv || !raw_ik || chunk <= 0 || offset < 0) return DSA_ERR_ARG;
    if (!st->pooled_kv || !st->pooled_ik || !st->rem_kv || !st->rem_ik) return DSA_ERR_ARG;
    if (!aligned16(raw_ik) || !aligned16(st->pooled_kv) || !aligned16(st->pooled_ik) ||
        !aligned16(st->rem_kv) || !aligned16(st->rem_ik))
        return DSA_ERR_ARG;
    const int32_t ratio = st->ratio;
    if (!valid_ratio(ratio)) return DSA_ERR_SHAPE;
    if (st->n_pooled_kv != st->n_pooled_ik) return DSA_ERR_DIVERGED;
    if (st->n_rem < 0 || st->n_rem >= ratio || st->n_pooled_kv < 0 ||
        st->n_pooled_kv * ratio + st->n_rem != st->n_tokens)
        return DSA_ERR_ARG;
    if (offset != st->n_tokens) return DSA_ERR_OFFSET;
    const int64_t end = offset + chunk;
    const int64_t n = end / ratio;
    if (n > st->cap) return DSA_ERR_CAPACITY;
    int rc = check_score_topk(q_idx, w, st->pooled_ik, n, chunk, offset, ratio, index_topk,
                              tile_rows, scratch, scratch_bytes, sel);
    if (rc != DSA_OK) return rc;
    rc = check_attention(q, raw_kv, raw_start, raw_rows, st->pooled_kv, n, sel, index_topk, chunk,
                         offset, ratio, window, scale, out);
    if (rc != DSA_OK) return rc;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const void *chunk_kv =
        static_cast<const uint8_t *>(raw_kv) + (offset - raw_start) * int64_t{kD} * 2;
    rc = launch_pool_append(*st, chunk_kv, raw_ik, chunk, offset, s);
    if (rc != DSA_OK) return rc;
    st->n_pooled_kv = st->n_pooled_ik = n;
    st->n_tokens = end;
    st->n_rem = static_cast<int32_t>(end % ratio);
    rc = run_score_topk(q_idx, w, st->pooled_ik, n, chunk, offset, ratio, index_topk, tile_rows,
                        scratch, sel, dev_status, s);
    if (rc != DSA_OK) return rc;
    return launch_attention(q, raw_kv, raw_start, raw_rows, st->pooled_kv, n, sel, index_topk,
                            chunk, offset, ratio, window, scale, out, dev_status, s);
}
