// The whole path for one chunk: pool/append, score + top-k (or the skip path),
// window + selected attention, enqueued in order on one stream with every
// argument checked before the first launch; and the same path from host
// buffers, with the host<->device copies overlapped with the kernels on a
// second stream.
//
// "perf(deepseek_v4): faster exact DeepSeek-V4 prefill", Summary (one prefill
// step per chunk; the compressor runs in every step) and "[Discussion] Tile
// indexed-attention scoring independently of the global prefill chunk",
// Possible design (a global chunk whose indexer work runs in bounded tiles).
#include "common.cuh"

namespace dsa {
namespace {

// Every argument of one chunk's path, checked before anything is enqueued.
int check_prefill(const dsa_pool_state *st, const void *raw_kv, int64_t raw_start,
                  int64_t raw_rows, const void *raw_ik, const void *q_idx, const float *w,
                  const void *q, int64_t chunk, int64_t offset, int32_t index_topk,
                  int32_t window, float scale, int64_t tile_rows, const void *scratch,
                  size_t scratch_bytes, const int32_t *sel, const void *out) {
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
    const int64_t n = (offset + chunk) / ratio;
    if (n > st->cap) return DSA_ERR_CAPACITY;
    int rc = check_score_topk(q_idx, w, st->pooled_ik, n, chunk, offset, ratio, index_topk,
                              tile_rows, scratch, scratch_bytes, sel);
    if (rc != DSA_OK) return rc;
    return check_attention(q, raw_kv, raw_start, raw_rows, st->pooled_kv, n, sel, index_topk,
                           chunk, offset, ratio, window, scale, out);
}

// The host-side state after this chunk's append. Written only once every launch
// of the call has been enqueued: a call that returns an error leaves it as it was.
void advance_state(dsa_pool_state *st, int64_t end) {
    st->n_pooled_kv = st->n_pooled_ik = end / st->ratio;
    st->n_tokens = end;
    st->n_rem = static_cast<int32_t>(end % st->ratio);
}

// Pool/append + score/top-k for one chunk on stream s (arguments checked, plan
// prepared); the state is advanced by the caller.
int enqueue_pool_and_select(const dsa_pool_state *st, const ScoreTopkPlan &plan,
                            const void *raw_kv, int64_t raw_start, const void *raw_ik,
                            const float *w, int64_t chunk, int64_t offset, int32_t index_topk,
                            int64_t tile_rows, void *scratch, int32_t *sel, int32_t *status,
                            cudaStream_t s) {
    const int32_t ratio = st->ratio;
    const int64_t n = (offset + chunk) / ratio;
    const void *chunk_kv =
        static_cast<const uint8_t *>(raw_kv) + (offset - raw_start) * int64_t{kD} * 2;
    int rc = launch_pool_append(*st, chunk_kv, raw_ik, chunk, offset, s);
    if (rc != DSA_OK) return rc;
    return enqueue_score_topk(plan, w, n, offset, ratio, index_topk, 0, chunk, tile_rows,
                              scratch, sel, status, s);
}

}  // namespace
}  // namespace dsa

extern "C" int dsa_prefill_chunk(dsa_pool_state *st, const void *raw_kv, int64_t raw_start,
                                 int64_t raw_rows, const void *raw_ik, const void *q_idx,
                                 const float *w, const void *q, int64_t chunk, int64_t offset,
                                 int32_t index_topk, int32_t window, float scale,
                                 int64_t tile_rows, void *scratch, size_t scratch_bytes,
                                 int32_t *sel, void *out, int32_t *dev_status, void *stream) {
    using namespace dsa;
    int rc = check_prefill(st, raw_kv, raw_start, raw_rows, raw_ik, q_idx, w, q, chunk, offset,
                           index_topk, window, scale, tile_rows, scratch, scratch_bytes, sel, out);
    if (rc != DSA_OK) return rc;
    const int64_t end = offset + chunk;
    const int64_t n = end / st->ratio;
    // everything that can fail short of a launch, before the first launch
    ScoreTopkPlan splan;
    AttnPlan aplan;
    rc = prepare_score_topk(q_idx, st->pooled_ik, n, chunk, index_topk, &splan);
    if (rc == DSA_OK) rc = prepare_attention(q, chunk, &aplan);
    if (rc != DSA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = enqueue_pool_and_select(st, splan, raw_kv, raw_start, raw_ik, w, chunk, offset,
                                 index_topk, tile_rows, scratch, sel, dev_status, s);
    if (rc == DSA_OK)
        rc = enqueue_attention(aplan, raw_kv, raw_start, st->pooled_kv, n, sel, index_topk, chunk,
                               offset, st->ratio, window, scale, out, dev_status, s);
    if (rc != DSA_OK) return rc;
    advance_state(st, end);
    return DSA_OK;
}

namespace {

struct Events {
    static constexpr int kMax = 16;
    cudaEvent_t e[kMax] = {};
    int n = 0;
    ~Events() {
        for (int i = 0; i < n; ++i) cudaEventDestroy(e[i]);  // released once complete
    }
    cudaEvent_t make() {
        if (n == kMax || cudaEventCreateWithFlags(&e[n], cudaEventDisableTiming) != cudaSuccess)
            return nullptr;
        return e[n++];
    }
};

}  // namespace

extern "C" int dsa_prefill_chunk_host(dsa_pool_state *st, const dsa_prefill_workspace *ws,
                                      const void *raw_kv_h, int64_t raw_start, int64_t raw_rows,
                                      const void *raw_ik_h, const void *q_idx_h, const float *w_h,
                                      const void *q_h, int64_t chunk, int64_t offset,
                                      int32_t index_topk, int32_t window, float scale,
                                      int64_t tile_rows, int32_t *sel_h, void *out_h,
                                      int32_t *dev_status, void *stream, void *copy_stream) {
    using namespace dsa;
    if (!ws || !raw_kv_h || !raw_ik_h || !q_idx_h || !w_h || !q_h || !sel_h || !out_h)
        return DSA_ERR_ARG;
    if (chunk > ws->max_chunk || index_topk > ws->max_topk || raw_rows > ws->raw_kv_rows)
        return DSA_ERR_CAPACITY;
    int rc = check_prefill(st, ws->raw_kv, raw_start, raw_rows, ws->raw_ik, ws->q_idx, ws->w,
                           ws->q, chunk, offset, index_topk, window, scale, tile_rows,
                           ws->scratch, ws->scratch_bytes, ws->sel, ws->out);
    if (rc != DSA_OK) return rc;
    const int64_t end = offset + chunk;
    const int64_t n = end / st->ratio;
    const size_t q_row = size_t{kH} * kD * 2;    // bytes of one query row (all heads)
    const size_t qi_row = size_t{kHI} * kDI * 2; // bytes of one indexer query row
    const size_t sel_row = size_t(index_topk) * 4;
    const int64_t sms = sm_count() > 0 ? sm_count() : 1;

    // every step's plan (tensor maps, per-device set-up), before the first copy or launch
    ScoreTopkPlan splan;
    rc = prepare_score_topk(ws->q_idx, st->pooled_ik, n, chunk, index_topk, &splan);
    if (rc != DSA_OK) return rc;

    // The indexer queries are the largest input the scoring waits for. The first score
    // tile is short (an eighth of the chunk), so it starts once its own rows have landed
    // while the rest copy on the other stream; the rows after it follow in tiles of
    // tile_rows. Results do not depend on the tiling. (At 4096 rows and 128K context a
    // first tile of 512 rows measured 3.82 ms end to end, 768 rows 3.85, 1024 rows 3.88,
    // 1536 rows 3.92.)
    int64_t first = std::min(tile_rows, chunk);
    if (splan.full && chunk >= 1024)
        first = std::min(first, std::max<int64_t>(256, (chunk / 8 + 127) / 128 * 128));

    // attention in row slices; each slice's output goes back while the next computes.
    // The output copy of a row takes about 0.95 of the kernel time of a row, so the
    // slices shrink towards the end by about that factor (whole waves of one row per
    // SM where possible): the copy left exposed after the last kernel is short and no
    // copy backlog builds up; the first slice is short enough that the output copies
    // start soon after the selection's. (At 4096 rows and 128K context these eight
    // slices measured 3.612 ms end to end against 3.652 for seven slices of 22, 19, 18,
    // 15, 11, 8 and 7 % of the rows.)
    int64_t cuts[8];
    int ncut = 0;
    {
        const int64_t waves = (chunk + sms - 1) / sms;
        static const double kCum[] = {0.185, 0.333, 0.481, 0.630, 0.741, 0.852, 0.926};
        if (chunk >= 1024) {
            for (double f : kCum) {
                const int64_t r = static_cast<int64_t>(f * static_cast<double>(waves) + 0.5) * sms;
                if (r > (ncut ? cuts[ncut - 1] : 0) && r < chunk) cuts[ncut++] = r;
            }
        }
        cuts[ncut++] = chunk;
    }
    AttnPlan aplan[8];
    for (int ci = 0; ci < ncut && rc == DSA_OK; ++ci) {
        const int64_t r0 = ci ? cuts[ci - 1] : 0;
        rc = prepare_attention(static_cast<const uint8_t *>(ws->q) + r0 * q_row, cuts[ci] - r0,
                               &aplan[ci]);
    }
    if (rc != DSA_OK) return rc;
    Events ev;
    cudaEvent_t in_done = ev.make(), qi_done = ev.make(), q_done = ev.make(),
                sel0_done = ev.make(), sel_done = ev.make(), all_done = ev.make();
    cudaEvent_t slice_done[8] = {};
    bool have_events = in_done && qi_done && q_done && sel0_done && sel_done && all_done;
    for (int ci = 0; ci < ncut; ++ci) have_events = have_events && (slice_done[ci] = ev.make());
    if (!have_events) return DSA_ERR_CUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStream_t c = static_cast<cudaStream_t>(copy_stream);
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
    const uint8_t *q_idx_hb = static_cast<const uint8_t *>(q_idx_h);
    uint8_t *q_idx_db = static_cast<uint8_t *>(ws->q_idx);
    uint8_t *sel_hb = reinterpret_cast<uint8_t *>(sel_h);
    const uint8_t *sel_db = reinterpret_cast<const uint8_t *>(ws->sel);
    bool ok = true;
    // inputs of pooling and the first score tile on the compute stream; the other
    // indexer query rows, then the attention queries, on the copy stream, landing while
    // pooling and the indexer run
    ok = ok && cudaMemcpyAsync(ws->raw_kv, raw_kv_h, size_t(raw_rows) * kD * 2, h2d, s) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(ws->raw_ik, raw_ik_h, size_t(chunk) * kDI * 2, h2d, s) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(ws->w, w_h, size_t(chunk) * kHI * 4, h2d, s) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(q_idx_db, q_idx_hb, size_t(first) * qi_row, h2d, s) == cudaSuccess;
    ok = ok && cudaEventRecord(in_done, s) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(c, in_done, 0) == cudaSuccess;
    if (first < chunk)
        ok = ok && cudaMemcpyAsync(q_idx_db + first * qi_row, q_idx_hb + first * qi_row,
                                   size_t(chunk - first) * qi_row, h2d, c) == cudaSuccess;
    ok = ok && cudaEventRecord(qi_done, c) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(ws->q, q_h, size_t(chunk) * q_row, h2d, c) == cudaSuccess;
    ok = ok && cudaEventRecord(q_done, c) == cudaSuccess;
    if (!ok) return DSA_ERR_CUDA;

    const void *chunk_kv =
        static_cast<const uint8_t *>(ws->raw_kv) + (offset - raw_start) * int64_t{kD} * 2;
    rc = launch_pool_append(*st, chunk_kv, ws->raw_ik, chunk, offset, s);
    if (rc == DSA_OK)
        rc = enqueue_score_topk(splan, ws->w, n, offset, st->ratio, index_topk, 0, first,
                                tile_rows, ws->scratch, ws->sel, dev_status, s);
    if (rc != DSA_OK) return rc;
    ok = ok && cudaEventRecord(sel0_done, s) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(s, qi_done, 0) == cudaSuccess;
    if (!ok) return DSA_ERR_CUDA;
    rc = enqueue_score_topk(splan, ws->w, n, offset, st->ratio, index_topk, first, chunk,
                            tile_rows, ws->scratch, ws->sel, dev_status, s);
    if (rc != DSA_OK) return rc;
    ok = ok && cudaEventRecord(sel_done, s) == cudaSuccess;
    // the selection goes back in two parts, the first while the later tiles score
    ok = ok && cudaStreamWaitEvent(c, sel0_done, 0) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(sel_hb, sel_db, size_t(first) * sel_row, d2h, c) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(c, sel_done, 0) == cudaSuccess;
    if (first < chunk)
        ok = ok && cudaMemcpyAsync(sel_hb + first * sel_row, sel_db + first * sel_row,
                                   size_t(chunk - first) * sel_row, d2h, c) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(s, q_done, 0) == cudaSuccess;
    if (!ok) return DSA_ERR_CUDA;

    for (int ci = 0; ci < ncut; ++ci) {
        const int64_t r0 = ci ? cuts[ci - 1] : 0;
        const int64_t rows = cuts[ci] - r0;
        rc = enqueue_attention(aplan[ci], ws->raw_kv, raw_start, st->pooled_kv, n,
                               ws->sel + r0 * index_topk, index_topk, rows, offset + r0,
                               st->ratio, window, scale,
                               static_cast<uint8_t *>(ws->out) + r0 * q_row, dev_status, s);
        if (rc != DSA_OK) return rc;
        ok = ok && cudaEventRecord(slice_done[ci], s) == cudaSuccess;
        ok = ok && cudaStreamWaitEvent(c, slice_done[ci], 0) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(static_cast<uint8_t *>(out_h) + r0 * q_row,
                                   static_cast<const uint8_t *>(ws->out) + r0 * q_row,
                                   size_t(rows) * q_row, d2h, c) == cudaSuccess;
        if (!ok) return DSA_ERR_CUDA;
    }
    ok = ok && cudaEventRecord(all_done, c) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(s, all_done, 0) == cudaSuccess;
    if (!ok) return DSA_ERR_CUDA;
    advance_state(st, end);
    return DSA_OK;
}
