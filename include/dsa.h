/*
 * dsa.h -- C ABI of libdsa.so: DeepSeek-V4 indexed sparse attention for a
 * chunked prefill on one GB300 GPU (sm_103a).
 *
 * The path has four steps, each a call below:
 *   (a) dsa_pool_append        ratio-4 mean pooling of the chunk's raw rows into
 *                              the PoolingCache, appended in place, remainder carried;
 *   (b,c) dsa_index_score_topk indexer scores of every query row against its
 *                              causally visible pooled rows (mask in the epilogue),
 *                              then per-row top-k, skipped when the pool fits;
 *   (d) dsa_window_sparse_attn exact attention over the raw sliding window plus
 *                              the selected pooled rows;
 *   dsa_prefill_chunk          the four steps for one chunk, in order;
 *   dsa_prefill_chunk_host     the same from host buffers, copies overlapped.
 *
 * Shapes are fixed by the model: indexer heads H_I=64 of dim d_I=128, query
 * heads H=64, one shared KV row of dim D=512 (key and value for every head),
 * B=1, bf16 storage, fp32 accumulation. The pooling ratio is a power of two
 * in [2, 128]: 4 for the indexed (sparse) attention, 128 for the compressed
 * attention whose selection is every visible pooled row (index_topk >= n).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers to row-major, densely packed
 *     arrays, 16-byte aligned (except the *_h arguments of
 *     dsa_prefill_chunk_host, which are host pointers). The library never allocates, frees or keeps a
 *     pointer after the call returns; the caller owns all memory.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Work is
 *     enqueued asynchronously; host-side state (dsa_pool_state counters) is
 *     updated at enqueue time, after the call's last launch or copy has been
 *     enqueued.
 *   - Every argument is validated, and every host-side step that can fail
 *     short of a launch (tensor-map encoding, per-device kernel set-up, event
 *     creation) is done, before anything is enqueued. On any such error the
 *     call returns a negative DSA_ERR_* code and changes nothing. The one
 *     exception is a launch or copy that the CUDA runtime rejects after earlier
 *     work of the same call was enqueued (DSA_ERR_CUDA; the context is then in
 *     an error state): the host-side state is still unchanged, but device
 *     memory written by the work already enqueued (for example the remainder
 *     rows of the pooling step) may have changed.
 *   - `dev_status` (optional, may be NULL) is a device int32 the kernels set
 *     to a DSA_ERR_* code when a bounded wait expires (DSA_ERR_TIMEOUT) or a
 *     gathered index is out of range (DSA_ERR_BOUNDS, the access is skipped).
 *     The caller zeroes it and reads it after synchronizing the stream.
 *
 * Notation: T = chunk rows; off = absolute position of the chunk's first
 * token; t = off + i for chunk row i; r = ratio; pooled row j covers raw
 * tokens j*r .. j*r+r-1 and is visible to t iff j*r+r-1 <= t, so
 * n_vis(t) = floor((t+1)/r); n = pooled rows after this chunk's append =
 * floor((off+T)/r).
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_RATIO 4
#define DSA_INDEX_HEADS 64
#define DSA_INDEX_DIM 128
#define DSA_HEADS 64
#define DSA_DIM 512

enum dsa_status {
    DSA_OK = 0,
    DSA_ERR_ARG = -1,       /* null pointer, non-positive size, misaligned pointer */
    DSA_ERR_SHAPE = -2,     /* bad ratio, index_topk <= 0, window <= 0, bad tile */
    DSA_ERR_OFFSET = -3,    /* offset != tokens already in the cache */
    DSA_ERR_CAPACITY = -4,  /* the append would exceed the preallocated cache */
    DSA_ERR_DIVERGED = -5,  /* KV and indexer caches hold different row counts */
    DSA_ERR_SCRATCH = -6,   /* scratch missing or smaller than required */
    DSA_ERR_CUDA = -7,      /* a CUDA launch or driver call failed */
    DSA_ERR_TIMEOUT = -8,   /* (device status) a bounded wait in a kernel expired */
    DSA_ERR_BOUNDS = -9,    /* (device status) an index was outside its buffer */
    DSA_ERR_RAW_RANGE = -10 /* raw KV buffer does not cover the window and chunk */
};

/*
 * PoolingCache of the two compressors (attention KV and indexer keys).
 * "perf(deepseek-v4): skip redundant all-pooled indexer scoring", Summary and
 * Correctness: both compressors run on every chunk, their pooled row counts
 * must agree, and a non-aligned prefill leaves a raw remainder (10 tokens at
 * ratio 4: two pooled rows, two raw rows left over). "perf(deepseek_v4):
 * faster exact DeepSeek-V4 prefill", Summary item 4: rows are appended in
 * place into a preallocated cache.
 *
 * Caller-owned host struct; the device buffers it points to are caller-owned:
 *   pooled_kv [cap, 512] bf16, pooled_ik [cap, 128] bf16,
 *   rem_kv    [ratio-1, 512] bf16, rem_ik [ratio-1, 128] bf16 (raw remainder rows,
 *             slot s = token n_pooled*ratio + s).
 * A fresh cache has all counters 0 and its ratio set. To resume from a prefix,
 * fill the first n_pooled rows and set n_tokens = n_pooled*ratio + n_rem.
 * Snapshot/rollback = copy this struct (and the n_rem remainder rows).
 */
typedef struct dsa_pool_state {
    void *pooled_kv;
    void *pooled_ik;
    void *rem_kv;
    void *rem_ik;
    int64_t cap;          /* rows allocated in pooled_kv and pooled_ik */
    int64_t n_pooled_kv;  /* pooled rows held in pooled_kv */
    int64_t n_pooled_ik;  /* pooled rows held in pooled_ik */
    int64_t n_tokens;     /* raw tokens consumed so far = absolute offset of the next chunk */
    int32_t n_rem;        /* raw remainder rows held (n_tokens mod ratio) */
    int32_t ratio;        /* raw tokens per pooled row: 4 (indexed) or 128 (compressed) */
} dsa_pool_state;

/*
 * (a) Pool and append one chunk.
 * Cites: the first page's Summary/Correctness (compressor runs once per chunk
 * in both paths; remainder); the second page's Summary item 4 (in-place append).
 * Reading taken: pooled row = mean of its `ratio` raw rows, summed in row
 * order in fp64 (exact for bf16 inputs of ordinary range), divided by the
 * ratio and rounded once to bf16 (round to nearest, ties to even).
 *
 *   raw_kv [chunk, 512] bf16, raw_ik [chunk, 128] bf16: the chunk's raw rows.
 *   chunk > 0; offset must equal st->n_tokens (else DSA_ERR_OFFSET);
 *   ratio must equal st->ratio, a power of two in [2, 128].
 * Writes pooled rows [n_old, n_new) of both caches and the new remainder, then
 * sets n_pooled_kv = n_pooled_ik = n_new = floor((offset+chunk)/ratio),
 * n_tokens = offset+chunk, n_rem = (offset+chunk) mod ratio.
 * Errors: DSA_ERR_ARG, DSA_ERR_SHAPE, DSA_ERR_OFFSET, DSA_ERR_CAPACITY
 * (n_new > cap), DSA_ERR_DIVERGED (n_pooled_kv != n_pooled_ik on entry), DSA_ERR_CUDA.
 */
int dsa_pool_append(dsa_pool_state *st, const void *raw_kv, const void *raw_ik,
                    int64_t chunk, int64_t offset, int32_t ratio, void *stream);

/*
 * Bytes of score scratch dsa_index_score_topk needs for tiles of `tile_rows`
 * query rows against `n_pooled` pooled rows: one fp32 score per (row, pooled
 * row), rows padded to a multiple of 128 pooled rows. "[Discussion] Tile
 * indexed-attention scoring independently of the global prefill chunk",
 * 128 GB / 1M-context motivation: the score buffer scales with rows x chunk
 * (4096 x 262,144 x 4 B = 4 GiB); Possible design: tiling bounds it by the
 * tile (1024 rows -> 1 GiB). Returns 0 for non-positive arguments.
 */
size_t dsa_score_scratch_bytes(int64_t tile_rows, int64_t n_pooled);

/*
 * (b)+(c) Indexer scores with the pooled-ratio causal mask, then top-k.
 * Cites: "perf(deepseek_v4): faster exact DeepSeek-V4 prefill", Summary item 5
 * (mask folded into the score epilogue) and Performance (all causally visible
 * pooled rows are scored); the first page's Summary (skip when every pooled row
 * fits within index_topk; empty and larger pools keep the full path); the
 * ds4 discussion, Possible design steps 1-5 (score/top-k in bounded query-row
 * tiles reusing one scratch).
 * Reading taken: s[t,j] = sum_{h<64} w[t,h] * ReLU(q_idx[t,h,:] . k[j,:]) for
 * j < n_vis(t), -inf otherwise; top-k order is (score desc, index asc); the
 * kept indices are written ascending and padded with -1.
 *
 *   q_idx [chunk, 64, 128] bf16; w [chunk, 64] fp32; pooled_ik [>= n_pooled, 128] bf16;
 *   n_pooled = n after this chunk's append; chunk > 0; offset >= 0 with
 *   n_pooled == floor((offset+chunk)/ratio); ratio a power of two in [2, 128];
 *   index_topk > 0;
 *   tile_rows > 0 (query rows per score/top-k tile; any value gives the same result);
 *   scratch: device buffer of scratch_bytes >= dsa_score_scratch_bytes(min(tile_rows,
 *   chunk), n_pooled) -- only touched on the full path (may be NULL otherwise);
 *   after the call it holds the last tile's scores, row-major with row stride
 *   round_up(n_pooled, 128) floats, masked entries -inf;
 *   sel [chunk, index_topk] int32 output.
 * Paths: n_pooled == 0 -> every sel entry -1 (no scoring);
 *        0 < n_pooled <= index_topk -> skip path: sel[i] = 0..n_vis(t)-1, -1 padded,
 *        q_idx/w/scratch are not read; otherwise the full path: rows with
 *        n_vis(t) <= index_topk keep all visible rows, the others their top index_topk.
 * Errors: DSA_ERR_ARG, DSA_ERR_SHAPE, DSA_ERR_SCRATCH, DSA_ERR_CUDA.
 */
int dsa_index_score_topk(const void *q_idx, const float *w, const void *pooled_ik,
                         int64_t n_pooled, int64_t chunk, int64_t offset, int32_t ratio,
                         int32_t index_topk, int64_t tile_rows, void *scratch,
                         size_t scratch_bytes, int32_t *sel, int32_t *dev_status,
                         void *stream);

/*
 * (d) Window + selected-pooled attention.
 * Cites: "perf(deepseek_v4): faster exact DeepSeek-V4 prefill", Summary item 1
 * (fused windowed + pooled prefill attention for B=1, H=64, D=512, bf16; the
 * kernel rebuilds causality, sliding window and pooled visibility from offsets)
 * and the ds4 discussion, Possible design step 4 (selected rows consumed by the
 * indexed attention).
 * Reading taken: for t and head h the keys are the raw rows
 * u = max(0, t-window+1) .. t followed by the selected pooled rows; each
 * 512-wide row is both key and value; logits = scale * q . row;
 * out = softmax-weighted sum of rows, accumulated in fp32, stored bf16.
 *
 *   q [chunk, 64, 512] bf16; raw_kv [raw_rows, 512] bf16 holding absolute raw
 *   rows raw_start .. raw_start+raw_rows-1, which must include
 *   max(0, offset-window+1) .. offset+chunk-1 (else DSA_ERR_RAW_RANGE);
 *   pooled_kv [>= n_pooled, 512] bf16; sel [chunk, index_topk] int32 as written
 *   by dsa_index_score_topk: row i holds min(index_topk, n_vis(t)) indices
 *   followed by -1 padding, and only those first min(index_topk, n_vis(t))
 *   entries are read; among them -1 is skipped, and an index outside
 *   [0, n_vis(t)) is skipped and reported as DSA_ERR_BOUNDS in dev_status;
 *   window > 0; scale > 0; out [chunk, 64, 512] bf16.
 * Launch shape: one 512-thread CTA per SM, each taking whole tokens; for a
 * chunk of at most (SM count / 8) rows whose tokens span more than one
 * 128-key block (decode steps, short bands), thread-block clusters of 8 CTAs
 * per token instead, merging their partial softmax results through
 * distributed shared memory (no memory beyond the arguments is used). The
 * result differs between the two shapes only by floating-point rounding.
 * Errors: DSA_ERR_ARG, DSA_ERR_SHAPE, DSA_ERR_RAW_RANGE, DSA_ERR_CUDA.
 */
int dsa_window_sparse_attn(const void *q, const void *raw_kv, int64_t raw_start,
                           int64_t raw_rows, const void *pooled_kv, int64_t n_pooled,
                           const int32_t *sel, int32_t index_topk, int64_t chunk,
                           int64_t offset, int32_t ratio, int32_t window, float scale,
                           void *out, int32_t *dev_status, void *stream);

/*
 * The whole path for one chunk: dsa_pool_append, dsa_index_score_topk,
 * dsa_window_sparse_attn, enqueued in that order on `stream`.
 * Cites: the second page's Summary (one fused prefill step per chunk); the
 * ds4 discussion, Possible design (global chunk with bounded indexer tiles).
 *
 *   raw_kv [raw_rows, 512] bf16 = absolute raw rows raw_start..; it must cover
 *   the window rows before the chunk and the chunk's own rows
 *   offset .. offset+chunk-1 (these are also what gets pooled);
 *   raw_ik [chunk, 128] bf16: the chunk's raw indexer-key rows;
 *   q_idx, w, q, scratch, sel, out: as in the calls above; offset must equal
 *   st->n_tokens.
 * On success the state is advanced as by dsa_pool_append.
 */
int dsa_prefill_chunk(dsa_pool_state *st, const void *raw_kv, int64_t raw_start,
                      int64_t raw_rows, const void *raw_ik, const void *q_idx,
                      const float *w, const void *q, int64_t chunk, int64_t offset,
                      int32_t index_topk, int32_t window, float scale, int64_t tile_rows,
                      void *scratch, size_t scratch_bytes, int32_t *sel, void *out,
                      int32_t *dev_status, void *stream);

/*
 * Device buffers for dsa_prefill_chunk_host, allocated and owned by the
 * caller (16-byte aligned device pointers). Capacities are in rows.
 */
typedef struct dsa_prefill_workspace {
    void *raw_kv;          /* [raw_kv_rows, 512] bf16 */
    int64_t raw_kv_rows;
    void *raw_ik;          /* [max_chunk, 128] bf16 */
    void *q_idx;           /* [max_chunk, 64, 128] bf16 */
    float *w;              /* [max_chunk, 64] fp32 */
    void *q;               /* [max_chunk, 64, 512] bf16 */
    int32_t *sel;          /* [max_chunk, max_topk] int32 */
    void *out;             /* [max_chunk, 64, 512] bf16 */
    void *scratch;         /* score scratch, see dsa_score_scratch_bytes */
    size_t scratch_bytes;
    int64_t max_chunk;
    int32_t max_topk;
} dsa_prefill_workspace;

/*
 * dsa_prefill_chunk for inputs and outputs in HOST memory: copies the chunk's
 * inputs to the workspace, runs the four steps and copies the selection and
 * the output back, overlapping the copies with the kernels.
 * The pages have no counterpart to this entry point: it is an addition of this
 * library (their prefill step starts from device-resident activations).
 *
 *   raw_kv_h [raw_rows, 512], raw_ik_h [chunk, 128], q_idx_h [chunk, 64, 128],
 *   w_h [chunk, 64] fp32, q_h [chunk, 64, 512]: host inputs with the meaning
 *   they have in dsa_prefill_chunk; sel_h [chunk, index_topk] int32 and
 *   out_h [chunk, 64, 512] bf16: host outputs. Pinned (page-locked) host
 *   memory is needed for the copies to overlap; pageable memory works but
 *   serializes them.
 *   ws: device buffers; chunk <= ws->max_chunk, index_topk <= ws->max_topk,
 *   raw_rows <= ws->raw_kv_rows, ws->scratch as for dsa_prefill_chunk.
 *   stream: the compute stream; copy_stream: a second stream for the copies
 *   that overlap compute (the query copy, the selection and output copies), or
 *   the same stream to serialize everything. Ordering: the inputs of pooling
 *   and of the first score tile (the chunk's first eighth of the indexer query
 *   rows) are copied on `stream`, the other indexer query rows and then the
 *   query rows on copy_stream while the pooling and indexer run; the later
 *   score tiles wait for their rows; the selection of the first tile is copied
 *   back while the later tiles score; the attention runs in up to eight row
 *   slices of shrinking size and each slice's output is copied back on
 *   copy_stream while the next slice computes. When `stream`
 *   completes, every copy has completed and the host outputs are valid.
 *   The host buffers must stay alive and unmodified until then.
 * Errors: those of dsa_prefill_chunk; DSA_ERR_ARG for a null host pointer or
 * workspace, DSA_ERR_CAPACITY when the chunk, index_topk or raw rows exceed
 * the workspace; DSA_ERR_CUDA if an event, copy or launch fails (the pool
 * state is advanced only once everything has been enqueued).
 */
int dsa_prefill_chunk_host(dsa_pool_state *st, const dsa_prefill_workspace *ws,
                           const void *raw_kv_h, int64_t raw_start, int64_t raw_rows,
                           const void *raw_ik_h, const void *q_idx_h, const float *w_h,
                           const void *q_h, int64_t chunk, int64_t offset, int32_t index_topk,
                           int32_t window, float scale, int64_t tile_rows, int32_t *sel_h,
                           void *out_h, int32_t *dev_status, void *stream, void *copy_stream);

/*
 * Library-held score scratch: the size of the device array that
 * dsa_index_score_topk_noalloc uses instead of a caller buffer (16 MiB, one
 * per device that loads the library, kept until the process exits).
 */
#define DSA_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * (b)+(c) as dsa_index_score_topk, for callers that cannot allocate device
 * memory when they call in -- for example code that only receives tensor
 * pointers from a host framework's execution loop, or a process that fixes its
 * device-memory budget at start-up and must not allocate while serving. The
 * score scratch is a file-scope device array inside libdsa.so
 * (DSA_STATIC_SCRATCH_BYTES); this call allocates nothing and frees nothing.
 * The pages have no counterpart to this entry point: it is an addition of this
 * library.
 *
 *   Arguments, paths and results are those of dsa_index_score_topk without
 *   `scratch` / `scratch_bytes`. On the full path the tile must fit the array:
 *   dsa_score_scratch_bytes(min(tile_rows, chunk), n_pooled) <= DSA_STATIC_SCRATCH_BYTES,
 *   otherwise DSA_ERR_SCRATCH is returned and nothing is enqueued (pick a
 *   smaller tile_rows; the selection does not depend on it).
 *   The first full-path call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) on the current device, and a later call looks it up
 *   again only if the device's context has changed (after cudaDeviceReset);
 *   make the first call on a device, and the first after a reset, before any
 *   stream capture.
 *   All calls on a device share the one array and it keeps the last call's
 *   contents (nothing in it needs to start at zero). Calls whose work overlaps
 *   on the GPU -- on different streams, or from several threads -- race on it;
 *   serialize them.
 * Errors: as dsa_index_score_topk; DSA_ERR_SCRATCH for a tile beyond the array;
 * DSA_ERR_CUDA if the array's address cannot be obtained.
 */
int dsa_index_score_topk_noalloc(const void *q_idx, const float *w, const void *pooled_ik,
                                 int64_t n_pooled, int64_t chunk, int64_t offset, int32_t ratio,
                                 int32_t index_topk, int64_t tile_rows, int32_t *sel,
                                 int32_t *dev_status, void *stream);

/*
 * Self-check of the error path behind DSA_ERR_TIMEOUT, for failure detection.
 * Every kernel of this library waits on shared-memory mbarriers with a bounded
 * wait: after about 2^31 SM cycles (about a second) it gives up, records
 * DSA_ERR_TIMEOUT in dev_status, lets the other warps of its CTA leave, and
 * the kernel returns, so the CUDA context stays usable. This call launches one
 * 32-thread CTA that initialises an mbarrier expecting one arrival and waits on
 * it with that same bounded wait:
 *   arrive != 0: a thread arrives first; the wait completes at once and
 *                dev_status is left as it is;
 *   arrive == 0: nothing arrives; about a second later DSA_ERR_TIMEOUT is
 *                written to dev_status (if it held DSA_OK) and the kernel ends.
 * dev_status: device int32, caller-owned. Enqueued on `stream`; returns
 * DSA_ERR_ARG for a null dev_status, DSA_ERR_CUDA if the launch fails.
 * The pages have no counterpart to this entry point: it is an addition of this
 * library.
 */
int dsa_bounded_wait_selftest(int32_t arrive, int32_t *dev_status, void *stream);

/* Static description of a DSA_* status code. */
const char *dsa_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H */
