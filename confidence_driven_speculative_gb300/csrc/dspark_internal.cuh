// dspark_internal.cuh -- device helpers and launch interfaces shared by the
// kernels of libdspark.so.  Not installed; the public interface is dspark.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

// ---------------------------------------------------------------------------
// Tuning constants.
// ---------------------------------------------------------------------------
constexpr int kThreads = 256;            // score / compact kernels: 256-thread CTAs
constexpr int kWarps = kThreads / 32;
constexpr int kConsumerWarps = 8;        // verify: consumer warps per CTA
constexpr int kVerifyThreads = (kConsumerWarps + 2) * 32;  // + producer and decider warps
constexpr int kChunkBytes = 16384;       // one vocab tile of one row (verify)
constexpr int kStages = 3;               // verify smem ring: kStages x (target + draft) tiles
constexpr int kSampleBlock = 4096;       // token ids per block of the two-level draw
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // bounded waits: 2 s (default)
constexpr uint64_t kDrainTimeoutNs = 100000000ull;  // a CTA that gave up waits this long at
                                                    // most for its own copies in flight

// Device status bits (workspace word 0).
constexpr int32_t kStatusWaitTimeout = 1;   // a wait on the shared-memory copy ring gave up
constexpr int32_t kStatusQueueTimeout = 2;  // a wait on other warps or CTAs (events, grid
                                            // barrier) gave up

// Draw modes of a request (DecideState::mode): the bonus draw from p at row
// L_b, the residual norm(max(0, p - q)) at row a_b, or p at the drawn row.
enum : int { D_BONUS = 0, D_RESID = 1, D_FALLBACK = 2 };

// Workspace q_ctr words shared by the small-batch verify and the tail kernel
// (the persistent verify uses words 0-9).
constexpr int kQTailExit = 10;   // tail CTAs exited
constexpr int kQSmallList = 11;  // rows listed for the tail kernel

// Per-request draw state written by the verify kernel's decide step.
struct DecideState {
    int a;                   // accepted drafts a_b
    int mode;                // 0 bonus (p at row L_b), 1 residual, 2 p at row a_b
    float Mp, Sp, Mq, Sq;    // normalisers of the drawn row (max, sum of 2^((z-max)s))
    float u_blk, u_tok;      // the draw's two uniforms
};


// ---------------------------------------------------------------------------
// Workspace layout (all offsets 256-byte aligned).
// ---------------------------------------------------------------------------
struct WorkspaceLayout {
    size_t status;        // int32
    size_t score_done;    // int32 [1]   hidden rows published
    size_t score_rows;    // int32 [1]   hidden rows claimed
    size_t verify_cnt;    // int32 [B]   per-request stream tiles done
    size_t r1_cnt;        // int32 [B]   per-request residual tiles done
    size_t bon_cnt;       // int32 [B]   per-request bonus-row tiles done
    size_t join;          // int32 [B]   drafts all accepted + bonus row streamed
    size_t rejflag;       // int32 [B]   launch epoch of a found rejection
    size_t q_ctr;         // int32 [16]  queue heads / tails, finished, exited, epoch, chunk,
                          //             audit totals
    size_t rowrec;        // float4 [B*(gamma+1) * nc]      row partials per (row, chunk)
    size_t blkrec;        // float2 [B * nblk * 8]          bonus-row block partials per warp
    size_t zrec;          // float2 [B * nblk * 8]          residual / p block masses per warp
    size_t gath;          // float2 [B * (gamma+1)]         z_p[d], z_q[d]
    size_t dstate;        // DecideState [B]
    size_t q_job;         // int2 [qcap]    residual-tile jobs (request, tile)
    size_t q_ready;       // int32 [qcap]
    size_t qb_job;        // int32 [2B]     decider jobs (decide / finish residual)
    size_t qb_ready;      // int32 [2B]
    size_t total;
    int nblk;             // sampling blocks per row
    int nc;               // 16 KB tiles per row (fp32, the larger count)
    int qcap;             // residual-tile queue capacity
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WorkspaceLayout workspace_layout(int B, int gamma, int V) {
    WorkspaceLayout w;
    const size_t rows = size_t(B) * size_t(gamma + 1);
    // fp32 rows need the most tiles; size for that so one workspace serves both dtypes
    w.nc = int((size_t(V) * 4 + kChunkBytes - 1) / kChunkBytes);
    w.nblk = (V + kSampleBlock - 1) / kSampleBlock;
    w.qcap = B * w.nc;  // per request at most one residual pass of nc tiles
    const size_t warps = kConsumerWarps;
    size_t off = 0;
    w.status = off;      off = align256(off + sizeof(int32_t));
    w.score_done = off;  off = align256(off + sizeof(int32_t));
    w.score_rows = off;  off = align256(off + sizeof(int32_t));
    w.verify_cnt = off;  off = align256(off + sizeof(int32_t) * size_t(B));
    w.r1_cnt = off;      off = align256(off + sizeof(int32_t) * size_t(B));
    w.bon_cnt = off;     off = align256(off + sizeof(int32_t) * size_t(B));
    w.join = off;        off = align256(off + sizeof(int32_t) * size_t(B));
    w.rejflag = off;     off = align256(off + sizeof(int32_t) * size_t(B));
    w.q_ctr = off;       off = align256(off + sizeof(int32_t) * 16);
    w.rowrec = off;      off = align256(off + 16 * rows * size_t(w.nc));
    w.blkrec = off;      off = align256(off + 8 * size_t(B) * w.nblk * warps);
    w.zrec = off;        off = align256(off + 8 * size_t(B) * w.nblk * warps);
    w.gath = off;        off = align256(off + 8 * rows);
    w.dstate = off;      off = align256(off + sizeof(DecideState) * size_t(B));
    w.q_job = off;       off = align256(off + 8 * size_t(w.qcap));
    w.q_ready = off;     off = align256(off + 4 * size_t(w.qcap));
    w.qb_job = off;      off = align256(off + 8 * size_t(B));
    w.qb_ready = off;    off = align256(off + 8 * size_t(B));
    w.total = off;
    return w;
}

// ---------------------------------------------------------------------------
// Element conversion.  bf16 -> fp32 is exact: the 16 bits become the top half.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T> struct Vec;
// 16-byte vector of 8 bf16 values
template <> struct Vec<uint16_t> {
    static constexpr int kElems = 8;
    static __device__ __forceinline__ void unpack(const uint4 &v, float (&x)[8]) {
        x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x);
        x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
        x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z);
        x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
    }
    static __device__ __forceinline__ float load1(const void *base, int64_t i) {
        const uint16_t h = static_cast<const uint16_t *>(base)[i];
        return __uint_as_float(uint32_t(h) << 16);
    }
};
// 16-byte vector of 4 fp32 values
template <> struct Vec<float> {
    static constexpr int kElems = 4;
    static __device__ __forceinline__ void unpack(const uint4 &v, float (&x)[4]) {
        x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
    }
    static __device__ __forceinline__ float load1(const void *base, int64_t i) {
        return static_cast<const float *>(base)[i];
    }
};

// 2^x on the SFU (MUFU.EX2); ftz flushes subnormal results, fine for
// softmax weights that are summed against a maximum of 1.
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------------------
// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11), written from the paper:
// per round two 64x64->128 products of counter words 0 and 2 with the two
// round multipliers; the new words are (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1,
// lo0); the key is bumped by two Weyl constants between rounds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void philox4x64_10(uint64_t (&c)[4], uint64_t k0, uint64_t k1) {
    const uint64_t m0 = 0xD2E7470EE14C6C93ull, m1 = 0xCA5A826395121157ull;
    const uint64_t w0 = 0x9E3779B97F4A7C15ull, w1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) { k0 += w0; k1 += w1; }
        const uint64_t hi0 = __umul64hi(m0, c[0]), lo0 = m0 * c[0];
        const uint64_t hi1 = __umul64hi(m1, c[2]), lo1 = m1 * c[2];
        const uint64_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
    }
}

// Uniforms of draft position k of request b: words 0, 1, 2 at counter
// (b, k, 0, 0) under key (seed, 0), each reduced to its top 24 bits / 2^24
// (exact in fp32): u (accept test), u_blk (block of a draw), u_tok (token
// within the block).
__device__ __forceinline__ void step_uniforms(uint64_t seed, int b, int k, float &u,
                                              float &u_blk, float &u_tok) {
    uint64_t c[4] = {uint64_t(b), uint64_t(k), 0ull, 0ull};
    philox4x64_10(c, seed, 0ull);
    u = float(uint32_t(c[0] >> 40)) * (1.0f / 16777216.0f);
    u_blk = float(uint32_t(c[1] >> 40)) * (1.0f / 16777216.0f);
    u_tok = float(uint32_t(c[2] >> 40)) * (1.0f / 16777216.0f);
}

// ---------------------------------------------------------------------------
// Online (max, sum) pairs in the base-2 domain: the pair (m, s) stands for
// sum_y 2^((z_y - m) * scale).  Combining rescales to the larger maximum.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ms_combine(float &m, float &s, float m2, float s2, float scale) {
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY) { m = mn; s = 0.f; return; }
    s = s * exp2_approx((m - mn) * scale) + s2 * exp2_approx((m2 - mn) * scale);
    m = mn;
}

__device__ __forceinline__ void warp_ms_reduce(float &m, float &s, float scale) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        ms_combine(m, s, m2, s2, scale);
    }
}

// (value, index) argmax; ties go to the lower index.
__device__ __forceinline__ void am_combine(float &v, int &i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i)) { v = v2; i = i2; }
}

__device__ __forceinline__ void warp_am_reduce(float &v, int &i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
        am_combine(v, i, v2, i2);
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ int warp_sum_int(int x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ---------------------------------------------------------------------------
// mbarrier + bulk TMA (cp.async.bulk, 1-D) in inline PTX.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// Global -> shared bulk copy; completion is signalled on `bar` as bytes.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Non-blocking test of phase `parity` of `bar`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar`, sleeping between polls once the wait
// has lasted a while: a warp that idles this way (a consumer with no tile
// coming) leaves its issue slots to the warps that still work.  Gives up
// after `limit_ns`.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (it >= 8) __nanosleep(it >= 64 ? 256u : 64u);
        if ((it & 15u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
    }
}

// Wait for phase `parity` of `bar`, giving up after `limit_ns`.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------------------
// Kernel argument blocks and launchers (defined in the .cu files).
// ---------------------------------------------------------------------------
struct ScoreArgs {
    int B, gamma, d;
    int hidden_bf16;
    const void *hidden;
    const float *head_w, *head_bias, *sts_tau;
    float cost_c;
    int cap_T;
    float *conf, *survival;
    int32_t *L0, *L, *draft_off, *row_off;
    int32_t *done_cnt, *row_ctr, *status;
    // Entropy-confidence variant: hidden points at the draft logits, d = V,
    // and ent_scale = log2(e) / theta.
    float ent_scale;
    uint64_t wait_ns;  // bound of every wait
    // pack != 0: the finishing CTA also writes the ragged packing (step a4)
    int pack;
    const int32_t *draft_tokens, *last_tokens, *seq_lens;
    int32_t *packed_ids, *packed_pos, *row_req, *row_k;
};

struct FixedArgs {
    int B, gamma, F;
    int32_t *L, *draft_off, *row_off;
    // pack != 0: also the ragged packing (step a4), one thread per slot
    int pack;
    const int32_t *draft_tokens, *last_tokens, *seq_lens;
    int32_t *packed_ids, *packed_pos, *row_req, *row_k;
};

struct CompactArgs {
    int B, gamma;
    const int32_t *L, *row_off, *draft_tokens, *last_tokens, *seq_lens;
    int32_t *packed_ids, *packed_pos, *row_req, *row_k;
};

struct VerifyArgs {
    int B, gamma, V;
    int nc;            // 16 KB tiles per row
    int chunk_elems;   // tokens per tile
    int elem_bytes;    // 2 (bf16) or 4 (fp32)
    int row_bytes;     // V * elem_bytes
    int nblk;          // sampling blocks per row
    int grp_stride;    // chunk slots per row in rowrec
    int qcap;          // residual-tile queue capacity
    int qbcap;         // decider queue capacity
    int greedy;
    float scale;       // log2(e) / Tm (sampling only)
    uint64_t seed;
    const int32_t *draft_tokens;
    const void *draft_logits, *target_logits;
    const int32_t *L, *draft_off, *row_off, *row_req, *row_k;
    int32_t *accept_len, *num_emitted, *out_tokens;
    float *p_tok, *q_tok;
    int32_t *seq_lens_commit;
    float4 *rowrec;
    float2 *blkrec, *zrec, *gath;
    DecideState *dstate;
    int2 *q_job;
    int32_t *q_ready, *q_ctr;
    int32_t *qb_job, *qb_ready;
    int32_t *req_cnt, *r1_cnt, *status;
    int32_t *bon_cnt, *join, *rejflag;
    // Cap-accept audit (all NULL on the plain verify): the window W_b that is
    // committed, the full-block acceptance a_b, and the batch totals.
    const int32_t *commit_len;
    int32_t *accept_full, *audit_totals;
    uint64_t wait_ns;  // bound of every wait
    // Small-batch verify with sampling: rejections are listed for the tail
    // kernel instead of drawn by the deciding CTA (rows of >= 4 tiles).
    int small_tail;
};

cudaError_t launch_score_budget(const ScoreArgs &a, int grid, cudaStream_t s);
int score_blocks_per_sm(int hidden_bf16);
cudaError_t launch_score_entropy(const ScoreArgs &a, int grid, cudaStream_t s);
int entropy_blocks_per_sm(int logit_bf16);
cudaError_t launch_fixed_budget(const FixedArgs &a, cudaStream_t s);
cudaError_t launch_compact(const CompactArgs &a, cudaStream_t s);
cudaError_t launch_verify(const VerifyArgs &a, int logit_bf16, int grid, cudaStream_t s);
// The residual rows of the requests the small-batch verify listed (row and
// draw state at q_job / dstate positions 0 .. q_ctr[kQSmallList]), in parts
// over the grid, and their draws; launched right after launch_verify_small.
int verify_tail_blocks_per_sm(int logit_bf16);
cudaError_t launch_verify_tail(const VerifyArgs &a, int logit_bf16, int grid, cudaStream_t s);
// The small-batch verify (verify_small.cu): which batches it takes, its row
// slices, and its launch.
constexpr int kSmallBatchMax = 16;
bool verify_small_fits(int B, int V, bool audit);
int verify_small_slices(int V);
cudaError_t launch_verify_small(const VerifyArgs &a, int logit_bf16, int grid, cudaStream_t s);
// The bound of every device wait in the next launches (0 restores kWaitTimeoutNs).
void set_wait_timeout_ns(uint64_t ns);
uint64_t wait_timeout_ns();
int verify_blocks_per_sm(int logit_bf16);
size_t verify_smem_bytes();

}  // namespace dspark
