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
// Keys of (t, h): raw rows u = max(0, t-W+1) .. t, then the first
// min(k, n_vis(t)) entries of sel[t, :] (entries that are -1 or outside
// [0, n_vis(t)) are skipped; the latter are reported). One 512-wide row is both
// key and value for all 64 heads.
//
// tcgen05 design, one token at a time per CTA (persistent over tokens), keys
// in blocks of 128 rows gathered with cp.async, everything transposed so the
// 128 keys sit on the MMA's M:
//   S^T[key, head]  = K_blk[128 x 512] . Q_t^T      (M=128, N=64, K=512)
//   O^T[d, head]   += V_blk^T[512 x 128] . P^T       (4 x (M=128, N=64, K=128))
// K_blk and V_blk are the same shared-memory tile (K = V): 8 chunks of
// [128 rows x 64 dims] with 128-byte swizzle, read K-major by the first MMA and
// MN-major by the second, filled and released in chunk pairs (one d-tile of
// the second MMA each) so the next block's rows stream in while PV drains; a
// ninth chunk slot takes chunk 7 of odd blocks so that chunk loads ahead.
// S^T (64 columns), O^T (4 x 64 columns) and the running max per head live in
// TMEM. Roles: six loader warps (key rows), one warp loading Q and issuing QK,
// one issuing PV, eight softmax warps that own TMEM lanes = keys: they mask,
// run the online softmax in the log2 domain (exp2 of scale*log2e*logit -
// running max) and write P^T as bf16. The running max is only raised when some
// logit exceeds it by more than 8 (log2 units): P then stays <= 256, and the
// rescale of O^T and of the partial sums is skipped on most blocks without
// changing the result (the same max divides out at the end). Output =
// O^T / sum, bf16, stored by the softmax warps straight from the registers they
// read O^T into.
//
// Few tokens (decode steps, short bands): one CTA per token would leave most SMs
// idle while it walks the token's blocks in sequence, so a cluster of 8 CTAs
// takes each token instead. CTA r takes blocks r, r+8, ... with its own online
// softmax; at the token's end the CTAs exchange (running max, sum) per head
// through distributed shared memory, scale their O^T by 2^(m_r - M) / L, stage
// it in their (now free) key tiles, and each sums one 64-dim slice of every head
// over the cluster. No global scratch is involved.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace dsa {

namespace {

// Warpgroups 0-1: loader warps 0-5, the QK-issuing warp 6 and the PV-issuing
// warp 7; warpgroups 2-3: softmax warps 8-15. setmaxnreg moves registers from
// the first two warpgroups to the softmax ones: 256*80 + 256*176 = 512*128, the
// launch allocation (checked on the host before the first launch).
//
// QK and PV are issued by two different warps: a thread that waits on an
// mbarrier between MMAs stalls its own issue until the MMAs it queued have been
// dispatched, so with one issuing thread every wait leaves the tensor pipe
// empty for a moment. With two, one warp's waits are covered by the other's
// queued MMAs.
constexpr int kLoadWarps = 6;
constexpr int kQkWarp = 6;
constexpr int kPvWarp = 7;
constexpr int kSoftWarp0 = 8;
constexpr int kAttnThreads = 512;
constexpr int kRegsLaunch = 128;
constexpr int kRegsLow = 80;
constexpr int kRegsSoft = 176;
constexpr int kSoftThreads = 256;
constexpr uint32_t kOffQ = 0;                 // 8 chunks x [64 heads x 128 B]
constexpr uint32_t kOffKV = 65536;            // 8 chunks x [128 keys x 128 B]
constexpr uint32_t kOffP = 65536 + 131072;    // P^T [128 keys x 64 heads] bf16
// A ninth key chunk slot: chunk 7 (dims 448..511) of odd blocks lives here, of even
// blocks in its usual slot, so a block's chunk 7 can land while the block before it
// still holds all eight usual slots; after the previous PV only chunk 6 is left to load.
constexpr uint32_t kOffX = kOffP + 16384;
// The per-block scratch of the rescale path and the per-token one of the epilogue are
// never live together (nor for the same heads), so they share space.
constexpr uint32_t kOffRed = kOffX + 16384;   // [4][64] block maxima  |  partial sums
constexpr uint32_t kOffLinv = kOffRed + 1024; // [64] rescale factors  |  1/sum
constexpr uint32_t kOffM = kOffLinv + 256;    // [2][64] running max (double-buffered)
constexpr uint32_t kOffBar = kOffM + 512;
constexpr uint32_t kAttnSmem = kOffBar + 256 + 1024;  // + slack for 1024-B alignment
static_assert(kAttnSmem <= 232448, "over the shared memory of one CTA");
constexpr uint32_t kLbo7Spare = kOffX - (kOffKV + 6 * 16384);  // chunk 6 -> spare chunk 7
constexpr uint32_t kSCol = 0;    // S^T: 2 x 64 TMEM columns (double-buffered by block parity)
constexpr uint32_t kOCol = 256;  // O^T: 4 d-tiles x 64 columns
// The running max of each head (log2 units), the same in all 128 lanes: 64 columns. A softmax
// thread loads its 32 heads' maxima together with the block's S^T under one wait, rather
// than with eight shared-memory loads per block (shared-memory instructions are the scarce
// issue resource of this kernel: its loaders' copies and the epilogue's stores use them too).
constexpr uint32_t kMCol = 128;
constexpr float kRescale = 8.0f;

struct AttnParams {
    __nv_bfloat16 *out;  // [T, 64, 512]
    const __nv_bfloat16 *raw_kv;
    const __nv_bfloat16 *pooled_kv;
    const int32_t *sel;
    int32_t k;
    int64_t n;
    int64_t offset;
    int64_t raw_start;
    int32_t ratio;
    int32_t window;
    float c;  // softmax scale * log2(e)
    int T;
    int32_t *status;
};

struct TokenInfo {
    int64_t t, nv, u0;
    int nwb, nsel, nb;
};

__device__ __forceinline__ TokenInfo token_info(const AttnParams &p, int i) {
    TokenInfo x;
    x.t = p.offset + i;
    x.nv = min(p.n, (x.t + 1) / p.ratio);
    x.u0 = max(int64_t{0}, x.t - p.window + 1);
    const int64_t nwin = x.t - x.u0 + 1;
    x.nwb = static_cast<int>((nwin + 127) / 128);
    x.nsel = static_cast<int>(min(static_cast<int64_t>(p.k), x.nv));
    x.nb = x.nwb + (x.nsel + 127) / 128;
    return x;
}

__device__ __forceinline__ float redux_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The softmax warps form two groups of four, one per half of the heads (named
// barriers 1 and 2, 128 threads each); barrier 3 spans all 256 softmax threads.
// OR of `pred` over the 128 threads of head group hh.
__device__ __forceinline__ bool vote_any_group(bool pred, int hh) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.b32 p, %1, 0;\n bar.red.or.pred q, %2, 128, p;\n"
        " selp.b32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(1 + hh)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void bar_group(int hh) {
    asm volatile("bar.sync %0, 128;" ::"r"(1 + hh) : "memory");
}

__device__ __forceinline__ void bar_soft() { asm volatile("bar.sync 3, 256;" ::: "memory"); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// tcgen05.mma / tcgen05.commit executed by every lane of a converged warp but
// issued only where `issue` is non-zero (one lane): the warp stays converged,
// so the operand descriptors can stay in uniform registers.
__device__ __forceinline__ void mma_bf16_if(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate, uint32_t issue) {
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %5, 0;\n"
        " @q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(issue)
        : "memory");
}

__device__ __forceinline__ void mma_commit_if(uint64_t *bar, uint32_t issue) {
    asm volatile(
        "{\n .reg .pred q;\n setp.ne.b32 q, %1, 0;\n"
        " @q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(
            smem_u32(bar)),
        "r"(issue)
        : "memory");
}

// Thread-block cluster helpers (the split mode below).
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_peer(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_peer4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Whether key block b is the last one this CTA takes of a token with nb blocks.
template <int kSplit>
__device__ __forceinline__ bool last_block(int b, int nb) {
    if constexpr (kSplit == 1) return b == nb - 1;
    else return b + kSplit >= nb;
}

// Every thread of every CTA of the cluster; orders shared-memory writes before it
// with reads after it, in any CTA of the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    const uint32_t b = smem_u32(bar);
    const long long t0 = clock64();
    while (!mbar_test(b, parity))
        if (clock64() - t0 > kWaitBudget) break;
}

// kSplit = 1: one CTA per token (persistent over tokens). kSplit > 1 (few tokens):
// a cluster of kSplit CTAs per token, CTA r taking the token's key blocks r,
// r + kSplit, ... with an online softmax of its own; at the token's end the
// cluster merges the partial results through distributed shared memory.
template <int kSplit>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem + kOffQ;
    uint8_t *sKV = smem + kOffKV;
    uint8_t *sP = smem + kOffP;
    float *sRed = reinterpret_cast<float *>(smem + kOffRed);
    float *sL = reinterpret_cast<float *>(smem + kOffRed);
    float *sLinv = reinterpret_cast<float *>(smem + kOffLinv);
    float *sM = reinterpret_cast<float *>(smem + kOffM);
    float *sAlpha = reinterpret_cast<float *>(smem + kOffLinv);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *q_full = bars + 0;
    uint64_t *q_free = bars + 1;
    uint64_t *kv_full = bars + 2;   // [4] chunk pairs 0-2, then chunk 6, landed
    uint64_t *x_full = bars + 6;    // [2] chunk 7 landed, by block parity (usual / spare slot)
    uint64_t *s_free = bars + 8;    // [2] S^T buffer read by the softmax, by block parity
    uint64_t *kv_free = bars + 10;  // [4] chunk pairs 0-2, then chunk 6, consumed by PV
    uint64_t *s_full = bars + 14;
    uint64_t *p_full = bars + 15;
    uint64_t *o_full = bars + 16;
    uint64_t *o_free = bars + 17;
    uint64_t *drain = bars + 18;    // [2] one per issuing warp

    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 21);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Each role walks tokens i0, i0 + istep, ... and of each the key blocks crank,
    // crank + kSplit, ... (read from special registers inside the roles, which keeps
    // them out of the register budget of the narrow warps).
#define DSA_SPLIT_COORDS                                                             \
    const int crank = kSplit > 1 ? static_cast<int>(cluster_rank()) : 0;             \
    const int i0 = static_cast<int>(blockIdx.x) / kSplit;                            \
    const int istep = static_cast<int>(gridDim.x) / kSplit;
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_free, 1);
        for (int m = 0; m < 4; ++m) mbar_init(&kv_full[m], 32 * kLoadWarps);  // noinc arrivals
        for (int m = 0; m < 4; ++m) mbar_init(&kv_free[m], 1);
        for (int q = 0; q < 2; ++q) {
            mbar_init(&x_full[q], 32 * kLoadWarps);
            mbar_init(&s_free[q], 8);  // one arrival per softmax warp
        }
        // a block's S^T is ready once its QK is done (QK warp) and the previous
        // block's PV no longer reads P or writes O^T (PV warp)
        mbar_init(s_full, 2);
        mbar_init(p_full, kSoftThreads);
        mbar_init(o_full, 1);
        mbar_init(o_free, 8);
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kPvWarp) tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp < kSoftWarp0) {
      // warpgroups 0-1 give registers to the softmax warpgroups (one instruction
      // instance for all eight warps)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
      if (warp < kLoadWarps) {
        // ---------------- loaders: key rows by cp.async (the QK warp loads Q), 8
        // lanes per 128-byte row piece, written straight into the 128-byte-swizzled tile.
        // Loader lw copies the 4-row groups lw, lw+6, lw+12, ... (at most 6, 24 rows).
        // Each block's selection entries are read one block ahead.
        DSA_SPLIT_COORDS
        const int lw = warp;
        const uint32_t kv_base = smem_u32(sKV);
        const uint32_t x_base = smem_u32(smem + kOffX);
        const int a = lane >> 3, pc = lane & 7;
        const int ngroups = (32 - lw + kLoadWarps - 1) / kLoadWarps;
        const bool holder = lane < 4 * ngroups;
        const int r_tile = 4 * (lw + kLoadWarps * (lane >> 2)) + (lane & 3);  // if holder
        auto fetch = [&](const TokenInfo &x, int i, int b) -> int32_t {
            const int pos = (b - x.nwb) * 128 + r_tile;
            return (holder && b >= x.nwb && pos < x.nsel)
                       ? __ldg(&p.sel[static_cast<int64_t>(i) * p.k + pos])
                       : -1;
        };
        auto row_of = [&](const TokenInfo &x, int b, int32_t j) -> int {
            if (b < x.nwb) {
                const int64_t u = min(x.u0 + 128 * b + r_tile, x.t);
                return static_cast<int>(u - p.raw_start);
            }
            const bool valid = j >= 0 && j < x.nv;
            const int pos = (b - x.nwb) * 128 + r_tile;
            if (holder && !valid && j != -1 && pos < x.nsel) report(p.status, DSA_ERR_BOUNDS);
            return valid ? j : 0;
        };
        int tok = 0, g = 0;
        bool ok = true;
        int i = i0;
        TokenInfo x = token_info(p, i < p.T ? i : 0);
        int32_t jn = i < p.T ? fetch(x, i, crank) : -1;
        for (; i < p.T && ok; i += istep, ++tok) {
            const int inext = i + istep;
            const TokenInfo xnext = token_info(p, inext < p.T ? inext : i);
            for (int b = crank; b < x.nb && ok; b += kSplit, ++g) {
                const int row = row_of(x, b, jn);
                const uint8_t *src_base =
                    reinterpret_cast<const uint8_t *>(b < x.nwb ? p.raw_kv : p.pooled_kv) + pc * 16;
                const int par = g & 1;
                // every group's source row, shuffled once for the block's eight chunks
                constexpr int kMaxGroups = (32 + kLoadWarps - 1) / kLoadWarps;
                int srows[kMaxGroups];
#pragma unroll
                for (int gq = 0; gq < kMaxGroups; ++gq)
                    srows[gq] = __shfl_sync(0xFFFFFFFFu, row, (4 * gq + a) & 31);
                // chunk 7 first, into the slot (usual one for even blocks, spare for odd
                // ones) of the block two back: this warp already waited for that block's
                // last PV tile before loading the previous block's chunk 6

#pragma unroll
                for (int gq = 0; gq < kMaxGroups; ++gq) {
                    if (gq >= ngroups) break;
                    const int r = 4 * (lw + kLoadWarps * gq) + a;
                    const int srow = srows[gq];
                    const uint8_t *src = src_base + static_cast<int64_t>(srow) * (kD * 2);
                    const uint32_t off = r * 128 + ((pc ^ (r & 7)) << 4);
                    cp_async16((par ? x_base : kv_base + 7 * 16384) + off, src + 7 * 128);
                }
                cp_async_arrive(&x_full[par]);
                jn = (b + kSplit < x.nb) ? fetch(x, i, b + kSplit)
                                         : (inext < p.T ? fetch(xnext, inext, crank) : -1);
                // chunk pairs 0-2, then chunk 6, as the previous block's PV releases them
                for (int m = 0; m < 4 && ok; ++m) {
                    if (lane == 0) ok = mbar_wait(&kv_free[m], (g & 1) ^ 1, abort_flag, p.status);
                    ok = (__ballot_sync(0xFFFFFFFFu, ok) & 1u) != 0;
                    if (!ok) break;
#pragma unroll
                    for (int gq = 0; gq < kMaxGroups; ++gq) {
                        if (gq >= ngroups) break;
                        const int r = 4 * (lw + kLoadWarps * gq) + a;
                        const int srow = srows[gq];
                        const uint8_t *src = src_base + static_cast<int64_t>(srow) * (kD * 2);
                        const uint32_t dst = kv_base + r * 128 + ((pc ^ (r & 7)) << 4);
                        cp_async16(dst + (2 * m) * 16384, src + (2 * m) * 128);
                        if (m < 3) cp_async16(dst + (2 * m + 1) * 16384, src + (2 * m + 1) * 128);
                    }
                    cp_async_arrive(&kv_full[m]);
                }
            }
            x = xnext;
        }
        // no copy into this CTA's shared memory may still be in flight at exit
        asm volatile("cp.async.wait_all;" ::: "memory");

        __syncwarp();
        if constexpr (kSplit > 1) {
            // the three cluster barriers of the softmax warps' merge
            cluster_sync();
            cluster_sync();
            cluster_sync();
        }
      } else if (warp == kQkWarp) {
        // ---------------- QK issuer (warp 6): S^T = K_blk . Q_t^T, chunk pair by chunk pair
        // as rows land. The whole warp runs the loop (descriptors stay warp-uniform) and
        // lane 0 issues: a lone diverged lane issues MMAs markedly slower.
        DSA_SPLIT_COORDS
        const uint32_t leader = lane == 0;
        constexpr uint32_t idesc_qk = idesc_bf16(128, 64, false, false);
        const uint64_t ad0 = desc_sw128(smem_u32(sKV), 16, 1024);
        const uint64_t adx = desc_sw128(smem_u32(smem + kOffX), 16, 1024);
        const uint64_t bd0 = desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t pol_stream = policy_evict_first();
        int tok = 0, g = 0, last_q = -1;
        bool ok = true;
        for (int i = i0; i < p.T && ok; i += istep, ++tok) {
            const TokenInfo x = token_info(p, i);
            // this token's queries: this warp's own QK of the previous token has read Q
            // (q_free), so the copy goes out as soon as that completes, without waiting for
            // the loaders
            if (!(ok = mbar_wait(q_free, (tok & 1) ^ 1, abort_flag, p.status))) break;
            if (leader) {
                mbar_expect_tx(q_full, 65536);
                for (int c = 0; c < 8; ++c)
                    tma_load_2d(sQ + c * 8192, &tm_q, q_full, c * 64, i * 64, pol_stream);
            }
            last_q = tok;
            if (!(ok = mbar_wait(q_full, tok & 1, abort_flag, p.status))) break;
            tc_fence_after();
            for (int b = crank; b < x.nb && ok; b += kSplit, ++g) {
                // S^T is double-buffered: the softmax of the block two back must have read
                // this buffer; then QK can start while the previous block's softmax runs
                const int par = g & 1;
                if (!(ok = mbar_wait(&s_free[par], ((g >> 1) & 1) ^ 1, abort_flag, p.status)))
                    break;
                const uint32_t s_col = tmem + kSCol + 64 * par;
                // chunk 7 landed early (usual slot on even blocks, spare slot on odd ones)
                if (!(ok = mbar_wait(&x_full[par], (g >> 1) & 1, abort_flag, p.status))) break;
                // rows landed through the generic proxy; the MMA reads via the async proxy
                fence_proxy_async_smem();
                tc_fence_after();
                {
                    const uint64_t ad = par ? adx : ad0 + ((7 * 16384) >> 4);
                    const uint64_t bd = bd0 + ((7 * 8192) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_if(s_col, ad + 2 * kk, bd + 2 * kk, idesc_qk, kk != 0,
                                    leader);
                }
#pragma unroll 1
                for (int m = 0; m < 4; ++m) {
                    // one wait per chunk pair (chunk 6 alone last): a wait stalls this warp's
                    // MMA issue
                    if (!(ok = mbar_wait(&kv_full[m], g & 1, abort_flag, p.status))) break;
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const uint64_t ad = ad0 + ((2 * m * 16384) >> 4);
                    const uint64_t bd = bd0 + ((2 * m * 8192) >> 4);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            if (m < 3 || h == 0)
                                mma_bf16_if(s_col, ad + ((h * 16384) >> 4) + 2 * kk,
                                            bd + ((h * 8192) >> 4) + 2 * kk, idesc_qk, 1u,
                                            leader);
                }
                if (!ok) break;
                mma_commit_if(s_full, leader);
                if (last_block<kSplit>(b, x.nb)) mma_commit_if(q_free, leader);
            }
        }
        mma_commit_if(&drain[0], leader);
        if (leader) drain_wait(&drain[0], 0);
        // no copy into this CTA's shared memory may still be in flight at exit
        if (leader && last_q >= 0) drain_wait(q_full, last_q & 1);
        __syncwarp();
        if constexpr (kSplit > 1) {
            cluster_sync();
            cluster_sync();
            cluster_sync();
        }
      } else {
        // ---------------- PV issuer (warp 7): O^T += V_blk^T . P^T, one d-tile at a time;
        // whole warp in the loop, lane 0 issues the 32 MMAs of a block in one straight run
        DSA_SPLIT_COORDS
        const uint32_t leader = lane == 0;
        constexpr uint32_t idesc_pv = idesc_bf16(128, 64, true, true);
        int tok = 0, g = 0;
        bool ok = true;
        if (leader) mbar_arrive(s_full);  // no PV precedes the first block
        __syncwarp();
        for (int i = i0; i < p.T && ok; i += istep, ++tok) {
            const TokenInfo x = token_info(p, i);
            for (int b = crank; b < x.nb && ok; b += kSplit, ++g) {
                if (!(ok = mbar_wait(p_full, g & 1, abort_flag, p.status))) break;
                tc_fence_after();
                if (b == crank && tok > 0) {
                    // the epilogue of the previous token must have read O^T
                    if (!(ok = mbar_wait(o_free, (tok - 1) & 1, abort_flag, p.status))) break;
                    tc_fence_after();
                }
                const uint32_t acc0 = b > crank;
                // d-tile 3 is chunks 6 and 7: on odd blocks chunk 7 sits in the spare slot
                const uint32_t lbo3 = (g & 1) ? kLbo7Spare : 16384u;
                if (leader) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_bf16(tmem + kOCol + 64 * m,
                                     desc_sw128(smem_u32(sKV + 2 * m * 16384 + kk * 2048),
                                                m < 3 ? 16384u : lbo3, 1024),
                                     desc_sw128(smem_u32(sP + kk * 2048), 8192, 1024), idesc_pv,
                                     kk > 0 ? 1u : acc0);
                        mma_commit(&kv_free[m]);
                    }
                }
                __syncwarp();
                mma_commit_if(s_full, leader);
                if (last_block<kSplit>(b, x.nb)) mma_commit_if(o_full, leader);
            }
        }
        mma_commit_if(&drain[1], leader);
        if (leader) drain_wait(&drain[1], 0);
        __syncwarp();
        if constexpr (kSplit > 1) {
            cluster_sync();
            cluster_sync();
            cluster_sync();
        }
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoft));
        // ---------------- softmax + epilogue, 8 warps: TMEM lanes of sub-partition sp
        // (keys, later dims) x heads [32*hh, 32*hh+32)
        DSA_SPLIT_COORDS
        const int st = threadIdx.x - 32 * kSoftWarp0;
        const int sp = warp & 3;
        const int hh = (warp - kSoftWarp0) >> 2;
        const int hb = 32 * hh;
        const int kl = sp * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(sp * 32) << 16);
        int tok = 0, g = 0, cur = 0;
        for (int i = i0; i < p.T; i += istep, ++tok) {
            const TokenInfo x = token_info(p, i);
            float l[32];
#pragma unroll
            for (int h = 0; h < 32; ++h) l[h] = 0.0f;
            if (sp == 0) sM[cur * 64 + hb + lane] = -INFINITY;
            {
                uint32_t ninf[32];
#pragma unroll
                for (int h = 0; h < 32; ++h) ninf[h] = __float_as_uint(-INFINITY);
                tmem_st32(lane_base + kMCol + hb, ninf);
                tmem_wait_st();
            }
            bar_group(hh);
            for (int b = crank; b < x.nb; b += kSplit, ++g) {
                bool valid;
                if (b < x.nwb) {
                    valid = x.u0 + 128 * b + kl <= x.t;
                } else {
                    const int pos = (b - x.nwb) * 128 + kl;
                    const int32_t j =
                        pos < x.nsel ? __ldg(&p.sel[static_cast<int64_t>(i) * p.k + pos]) : -1;
                    valid = j >= 0 && j < x.nv;
                }
                // S^T of this block is ready and the previous block's PV is done with P
                // and O^T
                const bool live = mbar_wait(s_full, g & 1, abort_flag, p.status);
                tc_fence_after();
                uint32_t sa[32], mv[32];
                tmem_ld32(lane_base + kMCol + hb, mv);
                if (live) tmem_ld32(lane_base + kSCol + 64 * (g & 1) + hb, sa);
                tmem_wait_ld();
                // this S^T buffer may take the QK of the block after next
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[g & 1]);
                valid = valid && live;
                // x = scale*log2e*logit - running max, once per (key, head); the same
                // values decide the rescale and feed exp2
                float xv[32];
                float xmax = -INFINITY;
                {
#pragma unroll
                    for (int h = 0; h < 32; ++h)
                        xv[h] = fmaf(__uint_as_float(sa[h]), p.c, -__uint_as_float(mv[h]));
                    float t16[16];
#pragma unroll
                    for (int h = 0; h < 16; ++h) t16[h] = fmaxf(xv[h], xv[h + 16]);
#pragma unroll
                    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                        for (int h = 0; h < w; ++h) t16[h] = fmaxf(t16[h], t16[h + w]);
                    xmax = t16[0];
                }
                if (vote_any_group(valid && xmax > kRescale, hh)) {
                    // exact block maxima -> new running max, then rescale sums and O^T
#pragma unroll
                    for (int h = 0; h < 32; ++h) {
                        const float wm =
                            redux_max(valid ? __uint_as_float(sa[h]) * p.c : -INFINITY);
                        if (lane == h) sRed[sp * 64 + hb + h] = wm;
                    }
                    bar_group(hh);
                    if (sp == 0) {
                        const int hd = hb + lane;
                        const float bm = fmaxf(fmaxf(sRed[hd], sRed[64 + hd]),
                                               fmaxf(sRed[128 + hd], sRed[192 + hd]));
                        const float m_old = sM[cur * 64 + hd];
                        const float m_new = fmaxf(m_old, bm);
                        sM[(cur ^ 1) * 64 + hd] = m_new;
                        sAlpha[hd] = ex2(m_old - m_new);
                    }
                    bar_group(hh);
                    cur ^= 1;
                    const float *m_now = sM + cur * 64 + hb;
#pragma unroll
                    for (int h = 0; h < 32; ++h) {
                        mv[h] = __float_as_uint(m_now[h]);
                        l[h] *= sAlpha[hb + h];
                        xv[h] = fmaf(__uint_as_float(sa[h]), p.c, -m_now[h]);
                    }
                    tmem_st32(lane_base + kMCol + hb, mv);
                    tmem_wait_st();
                    if (b > crank && live) {
#pragma unroll 1
                        for (int m = 0; m < 4; ++m) {
                            uint32_t oa[32];
                            const uint32_t col = lane_base + kOCol + 64 * m + hb;
                            tmem_ld32(col, oa);
                            tmem_wait_ld();
#pragma unroll
                            for (int h = 0; h < 32; ++h)
                                oa[h] = __float_as_uint(__uint_as_float(oa[h]) * sAlpha[hb + h]);
                            tmem_st32(col, oa);
                        }
                        tmem_wait_st();
                    }
                }
                // this thread's 32 heads of the P^T row for key kl: 4 swizzled 16-byte pieces.
                // The sums take P as rounded to bf16, the values the PV MMA multiplies, so
                // numerator and denominator weigh every key alike.
                {
                    float pr[32];
#pragma unroll
                    for (int h = 0; h < 32; ++h) pr[h] = valid ? ex2(xv[h]) : 0.0f;
                    uint8_t *prow = sP + kl * 128;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __nv_bfloat162 v =
                                __floats2bfloat162_rn(pr[8 * q + 2 * e], pr[8 * q + 2 * e + 1]);
                            pk[e] = *reinterpret_cast<const uint32_t *>(&v);
                            l[8 * q + 2 * e] += bf16lo(pk[e]);
                            l[8 * q + 2 * e + 1] += bf16hi(pk[e]);
                        }
                        *reinterpret_cast<uint4 *>(prow + (((4 * hh + q) ^ (kl & 7)) << 4)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(p_full);
            }
            // ---- token end: sums over keys, then O^T / sum -> out[t, h, d]
            // transpose-reduce the 32 partial sums across the warp: lane ends with
            // the warp's total for head hb + lane
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) {
                const bool hi = lane & 16;
                const float send = hi ? l[i2] : l[i2 + 16];
                const float keep = hi ? l[i2 + 16] : l[i2];
                l[i2] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
            }
#pragma unroll
            for (int i2 = 0; i2 < 8; ++i2) {
                const bool hi = lane & 8;
                const float send = hi ? l[i2] : l[i2 + 8];
                const float keep = hi ? l[i2 + 8] : l[i2];
                l[i2] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
            }
#pragma unroll
            for (int i2 = 0; i2 < 4; ++i2) {
                const bool hi = lane & 4;
                const float send = hi ? l[i2] : l[i2 + 4];
                const float keep = hi ? l[i2 + 4] : l[i2];
                l[i2] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 4);
            }
#pragma unroll
            for (int i2 = 0; i2 < 2; ++i2) {
                const bool hi = lane & 2;
                const float send = hi ? l[i2] : l[i2 + 2];
                const float keep = hi ? l[i2 + 2] : l[i2];
                l[i2] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 2);
            }
            {
                const bool hi = lane & 1;
                const float send = hi ? l[0] : l[1];
                const float keep = hi ? l[1] : l[0];
                l[0] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 1);
            }
            sL[sp * 64 + hb + lane] = l[0];
            if constexpr (kSplit == 1) {
                bar_soft();
                if (st < 64) sLinv[st] = 1.0f / (sL[st] + sL[64 + st] + sL[128 + st] + sL[192 + st]);
                bar_soft();
                // O^T (4 d-tiles x this warp's 32 heads) into registers one tile at a time, scaled
                // and stored straight to global memory: lane holds dim d = 128m + 32sp + lane of
                // heads hb..hb+31, so for each head the warp writes 32 consecutive dims (64
                // contiguous bytes). No staging in shared memory, so P's buffer stays free.
                const bool live = mbar_wait(o_full, tok & 1, abort_flag, p.status);
                tc_fence_after();
                __nv_bfloat16 *orow = p.out + (static_cast<int64_t>(i) * kH + hb) * kD + 32 * sp + lane;
                // this warp's 32 heads' 1/sum, read once for the four d-tiles (the store loop
                // is bound by its shared-memory and store instructions)
                float linv[32];
#pragma unroll
                for (int h = 0; h < 32; h += 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(&sLinv[hb + h]);
                    linv[h] = v.x;
                    linv[h + 1] = v.y;
                    linv[h + 2] = v.z;
                    linv[h + 3] = v.w;
                }
#pragma unroll 1
                for (int m = 0; m < 4; ++m) {
                    uint32_t oa[32];
                    if (live) {
                        tmem_ld32(lane_base + kOCol + 64 * m + hb, oa);
                        tmem_wait_ld();
                    }
                    if (live) {
                        __nv_bfloat16 *o = orow + 128 * m;
#pragma unroll
                        for (int h = 0; h < 32; ++h)
                            o[h * kD] = __float2bfloat16_rn(__uint_as_float(oa[h]) * linv[h]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_free);
            } else {
                // ---- merge of the cluster's partial results: CTA r holds, per head,
                // its running max m_r, sum l_r and O_r^T over its own blocks. With
                // M = max_r m_r and L = sum_r l_r 2^(m_r - M), the output is
                // sum_r O_r 2^(m_r - M) / L.
                const bool has = crank < x.nb;
                const bool live = has && mbar_wait(o_full, tok & 1, abort_flag, p.status);
                tc_fence_after();
                bar_soft();
                // P's buffer is free once the last PV is done: it carries (m_r, l_r)
                float *sXm = reinterpret_cast<float *>(sP);
                float *sXl = sXm + 64;
                if (st < 64) {
                    sXm[st] = has ? sM[cur * 64 + st] : -INFINITY;
                    sXl[st] = sL[st] + sL[64 + st] + sL[128 + st] + sL[192 + st];
                }
                cluster_sync();
                if (st < 64) {
                    float mr[kSplit], lr[kSplit];
                    float mx = -INFINITY;
#pragma unroll
                    for (int r = 0; r < kSplit; ++r) {
                        mr[r] = ld_peer(peer_addr(smem_u32(&sXm[st]), r));
                        lr[r] = ld_peer(peer_addr(smem_u32(&sXl[st]), r));
                        mx = fmaxf(mx, mr[r]);
                    }
                    float tot = 0.0f;
#pragma unroll
                    for (int r = 0; r < kSplit; ++r)
                        if (lr[r] > 0.0f) tot += lr[r] * ex2(mr[r] - mx);
                    sLinv[st] = sXl[st] > 0.0f ? ex2(sXm[st] - mx) / tot : 0.0f;
                }
                bar_soft();
                // this CTA's scaled O^T, fp32 [64 heads][512 dims], into its key tile
                // (free: the token's last PV is done and no token follows)
                float *stage = reinterpret_cast<float *>(sKV);
#pragma unroll 1
                for (int m = 0; m < 4; ++m) {
                    // (loaded even when this CTA ran no PV: a read of allocated but
                    // unwritten TMEM columns is harmless, and the value is dropped below)
                    uint32_t oa[32];
                    tmem_ld32(lane_base + kOCol + 64 * m + hb, oa);
                    tmem_wait_ld();
                    float *col = stage + hb * kD + 128 * m + 32 * sp + lane;
#pragma unroll
                    for (int h = 0; h < 32; ++h)
                        col[h * kD] = live ? __uint_as_float(oa[h]) * sLinv[hb + h] : 0.0f;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_free);
                cluster_sync();
                // dims [64 crank, 64 crank + 64) of every head: the sum over the cluster's
                // CTAs in rank order, rounded to bf16
                const uint32_t stage_u = smem_u32(stage);
#pragma unroll 1
                for (int it = st; it < kH * 16; it += kSoftThreads) {
                    const int h = it >> 4, q4 = it & 15;
                    const uint32_t off = static_cast<uint32_t>(h * kD + 64 * crank + 4 * q4) * 4u;
                    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                    for (int r = 0; r < kSplit; ++r) {
                        const float4 v = ld_peer4(peer_addr(stage_u + off, r));
                        acc.x += v.x;
                        acc.y += v.y;
                        acc.z += v.z;
                        acc.w += v.w;
                    }
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
                    uint2 pk;
                    pk.x = *reinterpret_cast<const uint32_t *>(&lo);
                    pk.y = *reinterpret_cast<const uint32_t *>(&hi);
                    *reinterpret_cast<uint2 *>(p.out + (static_cast<int64_t>(i) * kH + h) * kD +
                                               64 * crank + 4 * q4) = pk;
                }
                // no CTA leaves (or reuses its shared memory) while the others read it
                cluster_sync();
            }
        }
    }
#undef DSA_SPLIT_COORDS
    __syncthreads();
    if (warp == kPvWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// CTAs per token in the split mode (a portable cluster size).
constexpr int kSplitN = 8;

template <int kSplit>
int prepare_attention_kernel() {
    // the setmaxnreg split is only safe with the launch allocation it assumes
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, attn_kernel<kSplit>) != cudaSuccess ||
        fa.numRegs != kRegsLaunch)
        return DSA_ERR_CUDA;
    if (cudaFuncSetAttribute(attn_kernel<kSplit>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kAttnSmem) != cudaSuccess)
        return DSA_ERR_CUDA;
    return DSA_OK;
}

cudaLaunchConfig_t split_config(unsigned grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kAttnThreads, 1, 1);
    cfg.dynamicSmemBytes = kAttnSmem;
    cfg.stream = s;
    return cfg;
}

cudaLaunchAttribute cluster_attr() {
    cudaLaunchAttribute at = {};
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = kSplitN;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    return at;
}

}  // namespace

namespace {

// Per-device one-time set-up: the raised shared-memory limit of both kernel
// instances, and whether a cluster of kSplitN whole-SM CTAs can be resident.
struct AttnSetup {
    bool done = false;
    int rc = DSA_OK;
    bool split_ok = false;
};
std::mutex g_attn_mu;
AttnSetup g_attn_setup[kMaxDevices];

int attention_setup(bool *split_ok) {
    const int dev = current_device();
    if (dev < 0) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_attn_mu);
    AttnSetup &st = g_attn_setup[dev];
    if (!st.done) {
        st.rc = (prepare_attention_kernel<1>() == DSA_OK &&
                 prepare_attention_kernel<kSplitN>() == DSA_OK)
                    ? DSA_OK
                    : DSA_ERR_CUDA;
        if (st.rc == DSA_OK) {
            int nc = 0;
            cudaLaunchConfig_t cfg = split_config(kSplitN, nullptr);
            cudaLaunchAttribute at = cluster_attr();
            cfg.attrs = &at;
            cfg.numAttrs = 1;
            st.split_ok = cudaOccupancyMaxActiveClusters(&nc, attn_kernel<kSplitN>, &cfg) ==
                              cudaSuccess &&
                          nc > 0;
            (void)cudaGetLastError();
        }
        st.done = true;
    }
    *split_ok = st.split_ok;
    return st.rc;
}

}  // namespace

int prepare_attention(const void *q, int64_t chunk, AttnPlan *plan) {
    int rc = attention_setup(&plan->split_ok);
    if (rc != DSA_OK) return rc;
    if (!make_tmap_bf16(&plan->tm_q, q, kD, static_cast<uint64_t>(chunk) * kH, kD * 2, 64, 64))
        return DSA_ERR_CUDA;
    return DSA_OK;
}

int enqueue_attention(const AttnPlan &plan, const void *raw_kv, int64_t raw_start,
                      const void *pooled_kv, int64_t n, const int32_t *sel, int32_t k,
                      int64_t chunk, int64_t offset, int32_t ratio, int32_t window, float scale,
                      void *out, int32_t *status, cudaStream_t s) {
    AttnParams p;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.raw_kv = static_cast<const __nv_bfloat16 *>(raw_kv);
    p.pooled_kv = static_cast<const __nv_bfloat16 *>(pooled_kv);
    p.sel = sel;
    p.k = k;
    p.n = n;
    p.offset = offset;
    p.raw_start = raw_start;
    p.ratio = ratio;
    p.window = window;
    p.c = scale * 1.4426950408889634f;
    p.T = static_cast<int>(chunk);
    p.status = status;
    const int sms = std::max(1, sm_count());
    // key blocks of the chunk's last token (the most of any of its tokens)
    const int64_t t_last = offset + chunk - 1;
    const int64_t nv = std::min(n, (t_last + 1) / ratio);
    const int64_t nwin = t_last - std::max<int64_t>(0, t_last - window + 1) + 1;
    const int64_t nb = (nwin + 127) / 128 + (std::min<int64_t>(k, nv) + 127) / 128;
    if (plan.split_ok && chunk * kSplitN <= sms && nb > 1) {
        // few tokens: a cluster per token spreads its key blocks over kSplitN SMs
        cudaLaunchConfig_t cfg = split_config(static_cast<unsigned>(chunk * kSplitN), s);
        cudaLaunchAttribute at = cluster_attr();
        cfg.attrs = &at;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, attn_kernel<kSplitN>, plan.tm_q, p) != cudaSuccess)
            return DSA_ERR_CUDA;
        return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
    }
    const int grid = static_cast<int>(std::min<int64_t>(chunk, sms));
    attn_kernel<1><<<grid, kAttnThreads, kAttnSmem, s>>>(plan.tm_q, p);
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
    if (!valid_ratio(ratio) || k <= 0 || window <= 0 || !(scale > 0.0f) || isinf(scale))
        return DSA_ERR_SHAPE;
    if (chunk * kH > (int64_t{1} << 31) - 1 || raw_rows > (int64_t{1} << 31) - 1 ||
        n > (int64_t{1} << 31) - 1)
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
    AttnPlan plan;
    rc = prepare_attention(q, chunk, &plan);
    if (rc != DSA_OK) return rc;
    return enqueue_attention(plan, raw_kv, raw_start, pooled_kv, n_pooled, sel, index_topk, chunk,
                             offset, ratio, window, scale, out, dev_status,
                             static_cast<cudaStream_t>(stream));
}
