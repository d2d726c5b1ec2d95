// verify.cu -- steps a5-a6: streaming verify pass, accept / resample /
// bonus, commit.
//
// "DFlash to DSpark in SGLang", section "Background": the target checks all
// drafts in one forward, the accepted prefix is committed and the verify
// forward yields one bonus token.  "SGLang Integrates DSpark ...", section
// "The Old Problem with Speculative Decoding: It Breaks Down at Scale": the
// speculative-sampling rule (Chen et al. 2023) -- accept draft d with
// probability min(1, p(d)/q(d)); on the first rejection draw from
// norm(max(0, p - q)).  "DFlash to DSpark in SGLang", section "Serving
// DeepSeek-V4 with SGLang": speculation leaves the target distribution
// unchanged.
//
// Design (GB300).  The pass is HBM-bound: every packed target row (sum L + B)
// and every kept draft row (sum L) is read at most once, V logits each.
//
//  * One persistent grid, 2 CTAs per SM; each CTA is a producer
//    warp, 8 consumer warps and a decider warp.  The producer's lane 0 fills
//    a 3-stage shared-memory ring with 1-D bulk TMA copies (cp.async.bulk)
//    completing on "full" mbarriers with byte counts; each consumer warp
//    releases a stage on its "empty" mbarrier.  No block-wide barrier in the
//    loop.
//  * Stream work is a queue of chunks handed out by an atomic counter, in
//    two phases.  Phase P streams the decision rows (k < L_b: target row k
//    with draft row (b, k) in sampling) in packed-row order, whole rows and
//    then quarter rows for the last wave (single 16 KB tiles for small
//    batches).  Phase Q streams each request's bonus row (k = L_b), skipping
//    requests already known to reject: the method never reads past the
//    first rejection.
//  * A consumer warp owns one eighth of every tile.  For a pair row its
//    lanes keep (m, sum of 2^(z log2(e)/Tm - m)) accumulators for p and q
//    across the tiles of the chunk -- m a reference set by the lane's first
//    vector, raised only when a tile's terms would pass 2^64, so most
//    vectors cost no maximum -- and reduce once, at the chunk's
//    end, into a record slot of the row (plain stores: deterministic).  A
//    bonus row stores one slot per tile and warp, which gives the per-block
//    masses of the draw.  Greedy rows keep (max, lowest argmax).
//  * The producer books the stages it gets back: tiles are counted per
//    (request, decision / bonus) locally and published with one fenced
//    atomic per change.  A request whose decision rows are in becomes a
//    decide job; its bonus row being in, together with every draft accepted
//    (a join counter), makes the bonus-draw job.  Decider warps serve these
//    jobs from a device-wide queue.  A rejection queues residual-mass jobs
//    (one tile of the rejecting row pair, read again while it is still in
//    L2), served through the producers' rings: an idle decider warp claims
//    one and leaves its task in its CTA's shared-memory mailbox, which the
//    producer takes before its own chunks (so the producer's loop reads no
//    global word while it streams); a producer whose stream is done claims
//    from the queue itself.  The last of them queues the residual draw.
//  * Draws are two-level: a 4096-id block by mass (u'), then an id inside it
//    (u''); in-block running sums are fp32 over short lane runs combined in
//    two-float (TwoSum) arithmetic, as exact as fp64 on the fast fp32 pipe.
//  * Every wait is bounded (2 s) and sets a status bit when it gives up;
//    counters reset themselves at the end of the launch.
//  * The cap-accept audit arm ("DFlash to DSpark in SGLang", "The
//    confidence scheduler and verify modes") is the same launch with a
//    committed window W_b: every draft of the block is tested, the commit is
//    min(a_b, W_b), and a window that ends inside the accepted run draws
//    from p at row W_b through the residual-tile path (what compact's bonus
//    draw would be).
#include <climits>

#include "dspark_internal.cuh"

namespace dspark {
namespace {

constexpr int kCW = kConsumerWarps;
constexpr int kStageBytes = 2 * kChunkBytes;  // target tile + draft tile
constexpr size_t kSmemBytes = size_t(kStages) * kStageBytes;

enum : int { T_EXIT = 0, T_STREAM = 1, T_RESID = 2 };
// q_ctr words: residual-tile queue head / tail, finished requests, exited CTAs,
// launch epoch, stream-chunk counter, decide queue head / tail, audit sums.
enum : int { QA_HEAD = 0, QA_TAIL = 1, Q_FINISHED = 2, Q_EXITED = 3, Q_EPOCH = 4, Q_CHUNK = 5,
             QB_HEAD = 6, QB_TAIL = 7, Q_AFULL = 8, Q_ACOMMIT = 9 };

struct TaskInfo {
    int type;   // T_*
    int b;      // request
    int r;      // packed target row read by the stage
    int k;      // draft index of the draft row (pair) / of the drawn row
    int Lb;     // verify length of request b
    int j;      // tile index
    int g;      // stream: chunk slot of the row
    int y0;     // first token id of the stage
    int bytes;  // bytes per row in the stage
    int pair;   // a draft row sits in the second half of the stage
    int bytes2; // target-only rows: the row's next tile in the second half (0: none)
    int d;      // stream pair: drafted id (its gather target)
    int flush;  // stream: last tile of the chunk
    float Mp, Sp, Mq, Sq;  // residual: normalisers of the row pair (the decide's)
};

struct VSmem {
    uint64_t full[kStages], empty[kStages];
    TaskInfo task[kStages];
    float4 part[kStages][kCW];  // per-warp row partials of a chunk's last tile
    int done[kStages];          // warps finished with a chunk's last tile
    // A residual tile handed from the decider warp to the producer, so that
    // the producer reads no global word to find residual work while it
    // streams: mbox_full is 1 from the decider's write to the producer's take.
    TaskInfo mbox;
    int mbox_full;
};

// Grid-wide shape of the stream work, the same in every thread.  Two
// phases.  Phase P walks the packed rows and streams the decision rows
// (k < L_b; a bonus row's chunks are claimed and skipped): rows below nA are
// one chunk each, rows [nA, nB) are cut into chunks of Cb tiles (gprb per
// row), rows from nB on go out tile by tile.  Phase Q streams each
// request's bonus row (k = L_b) in chunks of CbQ tiles, skipping requests
// already known to reject.  So the accept tests -- and the residual draws
// they start -- run while the bonus rows are still streaming.
struct StreamShape {
    int n_rows;    // packed rows
    int nA;        // rows handed out whole
    int nB;        // first row handed out in single tiles
    int Cb;        // tiles per chunk in rows [nA, nB)
    int gprb;      // chunks per row in rows [nA, nB)
    int nq;        // chunks of rows [nA, nB)
    int nP;        // chunks of phase P
    int CbQ;       // tiles per chunk of a bonus row
    int gprbQ;     // chunks per bonus row
    int n_chunks;  // phase P and phase Q
};

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_relaxed(const int *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(int *p, int v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Release / acquire at GPU scope for the queues, books and join counters:
// with a relaxed store or atomic after it, a release pattern; with one
// before it, an acquire pattern.  Lighter than the sequentially consistent
// fence, which nothing here needs.
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
// q_ctr words 0-3 (residual head / tail, finished, exited) in one load.
__device__ __forceinline__ int4 ld_acquire_ctr4(const int *p) {
    int4 v;
    asm volatile("ld.acquire.gpu.global.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

// Cross-CTA state is read through L2 only (never a possibly stale L1 line).
__device__ __forceinline__ DecideState load_state(const VerifyArgs &a, int b) {
    static_assert(sizeof(DecideState) == 32, "two 16-byte loads");
    const int4 *p = reinterpret_cast<const int4 *>(a.dstate + b);
    const int4 lo = __ldcg(p), hi = __ldcg(p + 1);
    DecideState st;
    st.a = lo.x;
    st.mode = lo.y;
    st.Mp = __int_as_float(lo.z);
    st.Sp = __int_as_float(lo.w);
    st.Mq = __int_as_float(hi.x);
    st.Sq = __int_as_float(hi.y);
    st.u_blk = __int_as_float(hi.z);
    st.u_tok = __int_as_float(hi.w);
    return st;
}

__device__ __forceinline__ int verify_len(const VerifyArgs &a, int b) {
    return min(max(a.L[b], 0), a.gamma);
}

__device__ __forceinline__ StreamShape stream_shape(const VerifyArgs &a) {
    StreamShape sh;
    // packed rows as written by the compaction, never more than its capacity
    sh.n_rows = min(max(a.row_off[a.B], 0), a.B * (a.gamma + 1));
    const long long n_tiles = (long long)sh.n_rows * a.nc;
    if (n_tiles >= 32LL * gridDim.x) {
        // many rows: whole rows, then the last gridDim.x rows in quarters
        // (quarters everywhere, or single-tile chunks, cost more in chunk
        // overhead than they gain in balance)
        sh.nA = max(0, sh.n_rows - int(gridDim.x));
        sh.nB = sh.n_rows;
        sh.Cb = max(1, a.nc / 4);
        sh.CbQ = sh.Cb;
    } else {
        // few rows: single tiles
        sh.nA = 0;
        sh.nB = 0;
        sh.Cb = 1;
        sh.CbQ = 1;
    }
    sh.gprb = (a.nc + sh.Cb - 1) / sh.Cb;
    sh.nq = (sh.nB - sh.nA) * sh.gprb;
    sh.nP = sh.nA + sh.nq + (sh.n_rows - sh.nB) * a.nc;
    sh.gprbQ = (a.nc + sh.CbQ - 1) / sh.CbQ;
    sh.n_chunks = sh.nP + a.B * sh.gprbQ;
    return sh;
}

// Fold one vector of logits into a running (max, sum of 2^((z - max) * s)).
// The vector's terms are summed pairwise before joining the running sum.
template <int VE>
__device__ __forceinline__ void online_update(float &m, float &s, const float (&x)[VE],
                                              float scale) {
    float vm = x[0];
#pragma unroll
    for (int e = 1; e < VE; ++e) vm = fmaxf(vm, x[e]);
    if (vm > m) {
        s *= exp2_approx((m - vm) * scale);
        m = vm;
    }
    const float ms = m * scale;
    float t[VE];
#pragma unroll
    for (int e = 0; e < VE; ++e) t[e] = exp2_approx(fmaf(x[e], scale, -ms));
#pragma unroll
    for (int w = 1; w < VE; w <<= 1)
#pragma unroll
        for (int e = 0; e + w < VE; e += 2 * w) t[e] += t[e + w];
    s += t[0];
}

// One tile's share of a lane -- vectors v0 + lane + 32 i < v1 -- of NR rows
// folded into the lane's (m, s) pairs.  The pair (m, s) stands for
// sum 2^(z s - m) with m any reference, not necessarily the maximum: the
// lane's first vector of the chunk sets it, and later terms are summed
// against it without a running maximum.  A share whose sum exceeds 2^64 (a
// term far above the reference; inf or NaN included) is folded again with a
// running maximum, so every term stays below 2^64 relative to the reference
// and the sum is at least 1 (the reference's own term), as accurate as with
// the maximum.
template <typename T, int NR>
__device__ __forceinline__ void tile_fold(float (&m)[NR], float (&s)[NR],
                                          const uint4 *const (&xv)[NR], int v0, int v1,
                                          int lane, float scale) {
    constexpr int VE = Vec<T>::kElems;
    constexpr float kRefCap = 18446744073709551616.f;  // 2^64
    const int vb = v0 + lane;
    if (vb >= v1) return;
    float c[NR], ts[NR];
#pragma unroll
    for (int h = 0; h < NR; ++h) {
        if (m[h] == -INFINITY) {
            float x[VE];
            Vec<T>::unpack(xv[h][vb], x);
            float vm = x[0];
#pragma unroll
            for (int e = 1; e < VE; ++e) vm = fmaxf(vm, x[e]);
            m[h] = vm;
        }
        c[h] = -(m[h] * scale);
        ts[h] = 0.f;
    }
    for (int v = vb; v < v1; v += 32) {
#pragma unroll
        for (int h = 0; h < NR; ++h) {
            float x[VE], t[VE];
            Vec<T>::unpack(xv[h][v], x);
#pragma unroll
            for (int e = 0; e < VE; ++e) t[e] = exp2_approx(fmaf(x[e], scale, c[h]));
#pragma unroll
            for (int w = 1; w < VE; w <<= 1)
#pragma unroll
                for (int e = 0; e + w < VE; e += 2 * w) t[e] += t[e + w];
            ts[h] += t[0];
        }
    }
#pragma unroll
    for (int h = 0; h < NR; ++h) {
        if (ts[h] <= kRefCap) {
            s[h] += ts[h];
            continue;
        }
#pragma unroll 1
        for (int v = vb; v < v1; v += 32) {
            float x[VE];
            Vec<T>::unpack(xv[h][v], x);
            online_update<VE>(m[h], s[h], x, scale);
        }
    }
}

// Two-float numbers: the unevaluated sum hi + lo, |lo| <= ulp(hi) / 2.
// The draws' running sums use them instead of fp64, whose rate on this chip
// is a small fraction of fp32's: Knuth's TwoSum keeps each addition's
// rounding error, so sums of fp32 masses come out as exact as in fp64 while
// staying on the fp32 pipe (no contraction applies: there is no product).
struct F2 {
    float hi, lo;
};

__device__ __forceinline__ F2 f2(float x) { return F2{x, 0.f}; }

__device__ __forceinline__ F2 operator+(F2 a, F2 b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    const float e = (a.hi - (s - bb)) + (b.hi - bb) + (a.lo + b.lo);
    const float h = s + e;
    return F2{h, e - (h - s)};
}

__device__ __forceinline__ F2 operator-(F2 a, F2 b) { return a + F2{-b.hi, -b.lo}; }

// a * u for 0 <= u <= 1 (the product's error kept by an FMA)
__device__ __forceinline__ F2 f2_scale(F2 a, float u) {
    const float p = a.hi * u;
    const float e = fmaf(a.hi, u, -p) + a.lo * u;
    const float h = p + e;
    return F2{h, e - (h - p)};
}

__device__ __forceinline__ bool f2_gt(F2 a, F2 b) {
    return (a.hi - b.hi) + (a.lo - b.lo) > 0.f;
}

__device__ __forceinline__ F2 f2_shfl_up(F2 v, int o) {
    return F2{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}

__device__ __forceinline__ F2 f2_shfl(F2 v, int src) {
    return F2{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}

// Inclusive warp scan (lane order).  The two-float scans and sums run only
// in the draws and residual tiles; kept as loops, their code stays small,
// which measurably shortens the draw chains (that code is cold beside the
// consumers' hot loop and is fetched as it runs).
__device__ __forceinline__ F2 warp_scan_incl(F2 v, int lane) {
#pragma unroll 1
    for (int o = 1; o < 32; o <<= 1) {
        const F2 n = f2_shfl_up(v, o);
        if (lane >= o) v = v + n;
    }
    return v;
}

__device__ __forceinline__ F2 warp_sum_f2(F2 v) {
#pragma unroll 1
    for (int o = 16; o > 0; o >>= 1)
        v = v + F2{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
    return v;
}

// Two-float sum of eight floats, pairwise (three levels instead of a chain
// of eight).
__device__ __forceinline__ F2 sum8_f2(const float (&v)[kConsumerWarps]) {
    static_assert(kConsumerWarps == 8, "eight slots");
    const F2 a = (f2(v[0]) + f2(v[1])) + (f2(v[2]) + f2(v[3]));
    const F2 b = (f2(v[4]) + f2(v[5])) + (f2(v[6]) + f2(v[7]));
    return a + b;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---------------------------------------------------------------------------
// queues
// ---------------------------------------------------------------------------
// Residual-tile jobs (request b, tile c), served by every producer through
// its TMA ring.
__device__ void push_resid_jobs(const VerifyArgs &a, int b, int epoch) {
    const int pos = atomicAdd(&a.q_ctr[QA_TAIL], a.nc);
    for (int i = 0; i < a.nc; ++i)
        if (pos + i < a.qcap) a.q_job[pos + i] = make_int2(b, i);
    fence_acq_rel_gpu();  // every payload (and the caller's state) before any ready word
    for (int i = 0; i < a.nc; ++i)
        if (pos + i < a.qcap) st_relaxed(&a.q_ready[pos + i], epoch);
}

// Decider jobs, served by the decider warps: decide request b, or (with
// kFinishResidual / kBonusDraw set) finish its residual draw / make its
// bonus draw.
__device__ void push_decide(const VerifyArgs &a, int job, int epoch) {
    const int pos = atomicAdd(&a.q_ctr[QB_TAIL], 1);
    if (pos < a.qbcap) {
        a.qb_job[pos] = job;
        fence_acq_rel_gpu();
        st_relaxed(&a.qb_ready[pos], epoch);
    }
}

__device__ TaskInfo resid_task(const VerifyArgs &a, int2 jb) {
    TaskInfo t;
    t.type = T_RESID;
    t.b = jb.x;
    t.j = jb.y;
    t.d = -1;
    t.g = t.flush = 0;
    t.Lb = verify_len(a, t.b);
    const DecideState st = load_state(a, t.b);
    t.k = st.a;
    t.r = a.row_off[t.b] + st.a;
    t.Mp = st.Mp;
    t.Sp = st.Sp;
    t.Mq = st.Mq;
    t.Sq = st.Sq;
    t.pair = 1;
    t.y0 = t.j * a.chunk_elems;
    t.bytes = min(kChunkBytes, a.row_bytes - t.j * kChunkBytes);
    t.bytes2 = 0;
    return t;
}

// The CTA's residual-tile mailbox: one task, written by the decider warp's
// lane 0, taken by the producer.  The flag is read and written volatile;
// the block fences order the task's words against it on both sides.
__device__ __forceinline__ bool mbox_empty(VSmem &sm) {
    return *reinterpret_cast<volatile int *>(&sm.mbox_full) == 0;
}
__device__ __forceinline__ void mbox_put(VSmem &sm, const TaskInfo &t) {
    __threadfence_block();  // the slot was seen empty before it is written
    sm.mbox = t;
    __threadfence_block();  // the task before the flag
    *reinterpret_cast<volatile int *>(&sm.mbox_full) = 1;
}
__device__ __forceinline__ bool mbox_take(VSmem &sm, TaskInfo &t) {
    if (mbox_empty(sm)) return false;
    __threadfence_block();  // the flag before the task
    t = sm.mbox;
    __threadfence_block();  // the task read before the slot is freed
    *reinterpret_cast<volatile int *>(&sm.mbox_full) = 0;
    return true;
}

// ---------------------------------------------------------------------------
// producer: lane 0 of warp kCW
// ---------------------------------------------------------------------------
// The next chunk, fetched over several fills so that its global loads
// (counter, row ids, request metadata) never stall the issue of a tile.
struct ChunkFetch {
    // 0: claim an index, 1: row ids, 2: request data, 3: keep or skip,
    // 4: ready, 5: none left
    int stage;
    int c, q, r, g, b, k, Lb, d, rej;
};

__device__ __forceinline__ void fetch_step(const VerifyArgs &a, const StreamShape &sh,
                                           ChunkFetch &f, int epoch) {
    if (f.stage == 0) {
        f.c = int(gridDim.x) + atomicAdd(&a.q_ctr[Q_CHUNK], 1);
        f.stage = 1;
    } else if (f.stage == 1) {
        if (f.c >= sh.n_chunks) {
            f.stage = 5;
            return;
        }
        f.q = f.c >= sh.nP;
        if (f.q) {
            // phase Q: the bonus row of request b
            const int cc = f.c - sh.nP;
            f.b = cc / sh.gprbQ;
            f.g = cc - f.b * sh.gprbQ;
            f.r = a.row_off[f.b + 1] - 1;
            f.rej = ld_relaxed(&a.rejflag[f.b]);
        } else {
            if (f.c < sh.nA) {
                f.r = f.c;
                f.g = 0;
            } else if (f.c < sh.nA + sh.nq) {
                const int cc = f.c - sh.nA;
                f.r = sh.nA + cc / sh.gprb;
                f.g = cc - (f.r - sh.nA) * sh.gprb;
            } else {
                const int cc = f.c - sh.nA - sh.nq;
                f.r = sh.nB + cc / a.nc;
                f.g = cc - (f.r - sh.nB) * a.nc;
            }
            f.b = a.row_req[f.r];
            f.k = a.row_k[f.r];
            f.rej = 0;
        }
        f.stage = 2;
    } else if (f.stage == 2) {
        f.Lb = verify_len(a, f.b);
        if (f.q) {
            f.k = f.Lb;
            f.d = -1;
        } else {
            f.d = f.k < a.gamma ? a.draft_tokens[size_t(f.b) * a.gamma + f.k] : -1;
        }
        f.stage = 3;
    } else if (f.stage == 3) {
        // phase P skips bonus rows; phase Q skips requests already rejected
        const bool skip = f.q ? f.rej == epoch : f.k >= f.Lb;
        f.stage = skip ? 0 : 4;
    }
}

// Books of the stages the producer gets back: tiles are counted per
// (request, kind) locally and published with one fenced atomic per change.
// Decision-row tiles complete a request's decide job.  Bonus-row tiles
// complete its bonus row; the bonus draw then runs once the decide has
// accepted every draft (join counter), at once when there are no drafts.
// Residual tiles complete the request's residual masses and start the
// draw.  (Counted instead by a fenced atomic in each consumer warp, the
// residual tiles stalled the warps behind those fences.)
constexpr int kFinishResidual = 1 << 30;  // decider job: finish the residual draw
constexpr int kBonusDraw = 1 << 29;       // decider job: the bonus draw

// The count an atomic returned is checked one flush (or one fill) later, so
// the atomic's round trip overlaps the issue of copies instead of stalling it.
struct Books {
    int acc_b, acc_kind, acc_n, acc_total, acc_Lb;
    int chk_b, chk_kind, chk_end, chk_Lb, chk_old;  // a published count awaiting its check
};

// Act on the count published last: a completed request's job.
__device__ void check_books(const VerifyArgs &a, Books &bk, int epoch) {
    if (bk.chk_b < 0) return;
    const int b = bk.chk_b;
    if (bk.chk_old == bk.chk_end) {
        if (bk.chk_kind == 0) push_decide(a, b, epoch);
        else if (bk.chk_kind == 2) push_decide(a, b | kFinishResidual, epoch);
        else if (bk.chk_Lb == 0 || atomicAdd(&a.join[b], 1) == 1) push_decide(a, b | kBonusDraw, epoch);
    }
    bk.chk_b = -1;
}

__device__ void flush_books(const VerifyArgs &a, Books &bk, int epoch) {
    if (bk.acc_n == 0) return;
    check_books(a, bk, epoch);
    fence_acq_rel_gpu();
    const int b = bk.acc_b;
    int *cnt = bk.acc_kind == 0 ? a.req_cnt : bk.acc_kind == 1 ? a.bon_cnt : a.r1_cnt;
    bk.chk_old = atomicAdd(&cnt[b], bk.acc_n);
    bk.chk_b = b;
    bk.chk_kind = bk.acc_kind;
    bk.chk_end = bk.acc_total - bk.acc_n;  // the count before ours when ours completes it
    bk.chk_Lb = bk.acc_Lb;
    bk.acc_n = 0;
}

__device__ __forceinline__ void account(const VerifyArgs &a, Books &bk, const TaskInfo &t,
                                        int epoch) {
    if (t.type == T_EXIT) return;
    // 0: decision rows, 1: bonus row, 2: residual row
    const int kind = t.type == T_RESID ? 2 : t.k < t.Lb ? 0 : 1;
    if (t.b != bk.acc_b || kind != bk.acc_kind) {
        flush_books(a, bk, epoch);
        bk.acc_b = t.b;
        bk.acc_kind = kind;
        bk.acc_Lb = t.Lb;
        bk.acc_total = (kind == 0 ? t.Lb : 1) * a.nc;
    }
    bk.acc_n += t.bytes2 > 0 ? 2 : 1;
}

// Wait for every fill below `upto` to come back from the consumers and book it.
__device__ bool reclaim(const VerifyArgs &a, VSmem &sm, Books &bk, int &booked, int upto,
                        int epoch) {
    for (; booked < upto; ++booked) {
        const int s = booked % kStages;
        if (!mbar_wait_bounded(&sm.empty[s], (booked / kStages) & 1, a.wait_ns)) {
            atomicOr(a.status, kStatusWaitTimeout);
            return false;
        }
        account(a, bk, sm.task[s], epoch);
    }
    return true;
}

__device__ void producer(const VerifyArgs &a, VSmem &sm, uint8_t *ring, const StreamShape &sh,
                         int epoch, int pre_b, int pre_k) {
    ChunkFetch nextc;
    nextc.stage = 1;       // the first chunk is the CTA's own index; the counter
    nextc.c = blockIdx.x;  // hands out the rest from gridDim.x on
    if (int(blockIdx.x) < sh.nA && pre_b >= 0) {
        // Whole rows lead the stream, so that chunk is row blockIdx.x, whose
        // ids were loaded with the packed total.
        nextc.q = 0;
        nextc.r = blockIdx.x;
        nextc.g = 0;
        nextc.b = pre_b;
        nextc.k = pre_k;
        nextc.rej = 0;
        nextc.stage = 2;
    }
    int cr = 0, cg = 0, cb = 0, ck = 0, cLb = 0, cd = -1, cj = 0, cj_end = 0;
    bool in_chunk = false;
    Books bk{-1, 0, 0, 0, 0, -1, 0, 0, 0, 0};
    int booked = 0;
    // Residual tiles reach the producer through the CTA's mailbox, which the
    // decider warp fills (a global load in this loop would stall the issue
    // of a copy: with free stages a fill is shorter than an L2 round trip).
    // Once its stream is done the producer also claims from the queue itself.
    int pending = -1;  // a residual-queue index claimed by the producer
    for (int fill = 0;; ++fill) {
        TaskInfo t;
        t.type = T_EXIT;
        bool have = false, ok = true;
        // 1. residual tiles first
        if (mbox_take(sm, t)) have = true;
        // 2. then the stream chunks
        if (!have && !in_chunk) {
            while (nextc.stage < 4) fetch_step(a, sh, nextc, epoch);
            if (nextc.stage == 4) {
                cr = nextc.r;
                cg = nextc.g;
                cb = nextc.b;
                ck = nextc.k;
                cLb = nextc.Lb;
                cd = nextc.d;
                const int C = nextc.q ? sh.CbQ : cr < sh.nA ? a.nc : cr < sh.nB ? sh.Cb : 1;
                cj = cg * C;
                cj_end = min(a.nc, cj + C);
                in_chunk = true;
                nextc.stage = 0;
            }
        }
        if (!have && in_chunk) {
            t.type = T_STREAM;
            t.r = cr;
            t.g = cg;
            t.b = cb;
            t.k = ck;
            t.Lb = cLb;
            t.d = cd;
            t.j = cj;
            t.pair = !a.greedy && ck < cLb;
            t.y0 = cj * a.chunk_elems;
            t.bytes = min(kChunkBytes, a.row_bytes - cj * kChunkBytes);
            // a target-only row (greedy, or a bonus row) carries its next tile
            // in the stage's draft half: full stages whatever the row kind
            t.bytes2 = !t.pair && cj + 1 < cj_end
                           ? min(kChunkBytes, a.row_bytes - (cj + 1) * kChunkBytes) : 0;
            const int ntile = t.bytes2 > 0 ? 2 : 1;
            t.flush = cj + ntile == cj_end;
            cj += ntile;
            if (cj == cj_end) in_chunk = false;
            have = true;
        }
        // keep the next chunk coming; with many tiles of this chunk left, one
        // fetch stage every fourth fill, so its loads are back before use
        if (nextc.stage < 4 && (!in_chunk || cj_end - cj < 10 || (fill & 3) == 0))
            fetch_step(a, sh, nextc, epoch);
        // 3. nothing of our own left: book everything, then serve the
        //    residual queue until every request has finished
        if (!have) {
            ok = reclaim(a, sm, bk, booked, fill, epoch);
            flush_books(a, bk, epoch);
            check_books(a, bk, epoch);
            if (pending < 0) pending = atomicAdd(&a.q_ctr[QA_HEAD], 1);
            const uint64_t t0 = global_timer_ns();
            unsigned ns = 32;
            while (ok) {
                if (mbox_take(sm, t)) {
                    have = true;
                    break;
                }
                if (pending < a.qcap && ld_acquire(&a.q_ready[pending]) == epoch) {
                    t = resid_task(a, __ldcg(a.q_job + pending));
                    pending = -1;
                    have = true;
                    break;
                }
                if (ld_acquire(&a.q_ctr[Q_FINISHED]) >= a.B) break;
                if (global_timer_ns() - t0 > a.wait_ns) {
                    atomicOr(a.status, kStatusQueueTimeout);
                    break;
                }
                __nanosleep(ns);
                ns = min(ns * 2, 256u);
            }
        }
        // 4. take the stage back (booking what it held) and fill it
        const int s = fill % kStages;
        if (ok) ok = reclaim(a, sm, bk, booked, fill - kStages + 1, epoch);
        if (!ok) {
            // A wait gave up: let every copy still in flight land (each is
            // the only outstanding use of its stage) before the CTA can
            // leave.  The consumers give up on their own waits.
            for (int f = booked; f < fill; ++f)
                mbar_wait_bounded(&sm.full[f % kStages], (f / kStages) & 1, kDrainTimeoutNs);
            return;
        }
        if (!have) t.type = T_EXIT;
        sm.task[s] = t;
        if (t.type == T_EXIT) {
            mbar_arrive(&sm.full[s]);
            return;
        }
        uint8_t *dst = ring + s * kStageBytes;
        uint64_t *bar = &sm.full[s];
        const char *tsrc = static_cast<const char *>(a.target_logits) +
                           size_t(t.r) * a.row_bytes + size_t(t.y0) * a.elem_bytes;
        mbar_arrive_expect_tx(bar, uint32_t(t.bytes) * (t.pair ? 2u : 1u) + uint32_t(t.bytes2));
        bulk_g2s(dst, tsrc, uint32_t(t.bytes), bar);
        if (t.pair) {
            const char *dsrc = static_cast<const char *>(a.draft_logits) +
                               (size_t(t.b) * a.gamma + t.k) * size_t(a.row_bytes) +
                               size_t(t.y0) * a.elem_bytes;
            bulk_g2s(dst + kChunkBytes, dsrc, uint32_t(t.bytes), bar);
        } else if (t.bytes2 > 0) {
            bulk_g2s(dst + kChunkBytes, tsrc + kChunkBytes, uint32_t(t.bytes2), bar);
        }
        // 5. act on the count published last, then book whatever has already
        //    come back, without waiting
        check_books(a, bk, epoch);
        while (booked < fill && mbar_test_wait(&sm.empty[booked % kStages], (booked / kStages) & 1)) {
            account(a, bk, sm.task[booked % kStages], epoch);
            ++booked;
        }
    }
}

// ---------------------------------------------------------------------------
// decisions (warp-level)
// ---------------------------------------------------------------------------
// Draft tokens d_{b, lane} and d_{b, lane + 32} of a request, loaded once per
// decision (gamma <= 64).
// (lane 0 also holds the request's cached length, loaded with the drafts so
// that the commit at the end of the chain is a store, not a round trip)
struct Drafts {
    int t[2];
    int seq;
};

__device__ __forceinline__ Drafts load_drafts(const VerifyArgs &a, int b, int lane) {
    Drafts d;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int k = lane + 32 * i;
        d.t[i] = k < a.gamma ? __ldcg(a.draft_tokens + size_t(b) * a.gamma + k) : -1;
    }
    d.seq = lane == 0 && a.seq_lens_commit ? __ldcg(a.seq_lens_commit + b) : 0;
    return d;
}

__device__ void finish_request(const VerifyArgs &a, int b, int acc, int token, const Drafts &dr,
                               int lane) {
    const int g1 = a.gamma + 1;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const int j = lane + 32 * i;
        if (j >= g1) continue;
        int v = -1;
        if (j < acc) v = dr.t[i < 2 ? i : 1];
        else if (j == acc) v = token;
        a.out_tokens[size_t(b) * g1 + j] = v;
    }
    if (lane == 0) {
        a.accept_len[b] = acc;
        a.num_emitted[b] = acc + 1;
        if (a.seq_lens_commit) a.seq_lens_commit[b] = dr.seq + acc + 1;
        a.req_cnt[b] = 0;
        a.r1_cnt[b] = 0;
    }
    // No fence: nothing in the kernel reads the outputs; the count only
    // tells the waiting warps when to leave, and the kernel's end publishes
    // the outputs.
    __syncwarp();
    if (lane == 0) atomicAdd(&a.q_ctr[Q_FINISHED], 1);
}

// Choose a sampling block: the smallest i whose running mass exceeds
// u * total; the last block with positive mass if rounding leaves no
// crossing.  mass(i) is evaluated by the lane that owns i.  Up to 64
// blocks, each lane's masses are evaluated once and the total is the last
// running mass (so it agrees with the scan exactly); more blocks take two
// sweeps.
template <typename F>
__device__ int choose_block(int nblk, float u, F mass, int lane) {
    if (nblk <= 64) {
        const F2 m0 = lane < nblk ? mass(lane) : f2(0.f);
        const F2 m1 = lane + 32 < nblk ? mass(lane + 32) : f2(0.f);
        const F2 i0 = warp_scan_incl(m0, lane);
        F2 i1 = f2(0.f), total = f2_shfl(i0, 31);
        if (nblk > 32) {
            i1 = total + warp_scan_incl(m1, lane);
            total = f2_shfl(i1, 31);
        }
        const F2 target = f2_scale(total, u);
        unsigned hit = __ballot_sync(0xffffffffu, lane < nblk && f2_gt(i0, target));
        if (hit) return __ffs(hit) - 1;
        hit = __ballot_sync(0xffffffffu, lane + 32 < nblk && f2_gt(i1, target));
        if (hit) return 32 + __ffs(hit) - 1;
        unsigned pos = __ballot_sync(0xffffffffu, lane + 32 < nblk && m1.hi > 0.f);
        if (pos) return 32 + 31 - __clz(pos);
        pos = __ballot_sync(0xffffffffu, lane < nblk && m0.hi > 0.f);
        return pos ? 31 - __clz(pos) : 0;
    }
    F2 total = f2(0.f);
    for (int t0 = 0; t0 < nblk; t0 += 32) {
        const int i = t0 + lane;
        total = total + warp_sum_f2(i < nblk ? mass(i) : f2(0.f));
    }
    const F2 target = f2_scale(total, u);
    F2 run = f2(0.f);
    int last_pos = 0;
    for (int t0 = 0; t0 < nblk; t0 += 32) {
        const int i = t0 + lane;
        const F2 v = i < nblk ? mass(i) : f2(0.f);
        const F2 incl = run + warp_scan_incl(v, lane);
        const unsigned hit = __ballot_sync(0xffffffffu, i < nblk && f2_gt(incl, target));
        if (hit) return t0 + __ffs(hit) - 1;
        const unsigned pos = __ballot_sync(0xffffffffu, i < nblk && v.hi > 0.f);
        if (pos) last_pos = t0 + 31 - __clz(pos);
        run = f2_shfl(incl, 31);
    }
    return last_pos;
}

// Draw weights of the VE elements of 16-byte vector v: 2^((z - Mp) s) for a
// draw from p (bonus, fallback); max(0, p - q) for the residual.
template <typename T>
__device__ __forceinline__ void draw_weights(const uint4 *tv, const uint4 *dv, int v, int mode,
                                             float Mp, float iSp, float Mq, float iSq,
                                             float scale, float (&w)[Vec<T>::kElems]) {
    constexpr int VE = Vec<T>::kElems;
    float x[VE];
    Vec<T>::unpack(__ldcg(tv + v), x);
    if (mode == D_RESID) {
        float y[VE];
        Vec<T>::unpack(__ldcg(dv + v), y);
#pragma unroll
        for (int e = 0; e < VE; ++e)
            w[e] = fmaxf(0.f, exp2_approx((x[e] - Mp) * scale) * iSp -
                                  exp2_approx((y[e] - Mq) * scale) * iSq);
    } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) w[e] = exp2_approx((x[e] - Mp) * scale);
    }
}

template <int VE>
__device__ __forceinline__ float pair_sum(const float (&w)[VE]) {
    float t[VE];
#pragma unroll
    for (int e = 0; e < VE; ++e) t[e] = w[e];
#pragma unroll
    for (int s = 1; s < VE; s <<= 1)
#pragma unroll
        for (int e = 0; e + s < VE; e += 2 * s) t[e] += t[e + s];
    return t[0];
}

// The token of a draw inside one slot -- the ids [y0, y0 + n) that one
// consumer warp covers in a tile: the smallest id whose running weight,
// counted from the slot's start, exceeds `target`.  Each lane owns a
// contiguous run of n/32 ids (kRunVec 16-byte vectors, one batch of loads);
// per-vector weights are summed pairwise and kept in registers; runs are
// combined in two-float sums; the lane holding the crossing finds its vector from the
// kept sums and reloads only that vector.  If rounding leaves no crossing,
// the last id with positive weight.  The rows were streamed moments
// earlier, so the loads hit L2.
template <typename T>
__device__ int slot_pick(const VerifyArgs &a, const DecideState &st, int b, int r, int y0, int n,
                         F2 target, int lane) {
    constexpr int VE = Vec<T>::kElems;
    constexpr int kRunVec = 4;  // n = 32 lanes x 4 vectors (1024 bf16 / 512 fp32 ids)
    const uint4 *tv = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.target_logits) +
                                                      size_t(r) * a.row_bytes);
    const uint4 *dv = reinterpret_cast<const uint4 *>(
        static_cast<const char *>(a.draft_logits) + (size_t(b) * a.gamma + st.a) * a.row_bytes);
    const int v_end = min(a.row_bytes / 16, (y0 + n) / VE);
    const float scale = a.scale, iSp = 1.f / st.Sp, iSq = 1.f / st.Sq;
    const bool resid = st.mode == D_RESID;
    const int v0 = y0 / VE + lane * kRunVec;
    auto weights = [&](const uint4 &xv, const uint4 &yv, float (&w)[VE]) {
        float x[VE];
        Vec<T>::unpack(xv, x);
        if (resid) {
            float y[VE];
            Vec<T>::unpack(yv, y);
#pragma unroll
            for (int e = 0; e < VE; ++e)
                w[e] = fmaxf(0.f, exp2_approx((x[e] - st.Mp) * scale) * iSp -
                                      exp2_approx((y[e] - st.Mq) * scale) * iSq);
        } else {
#pragma unroll
            for (int e = 0; e < VE; ++e) w[e] = exp2_approx((x[e] - st.Mp) * scale);
        }
    };
    uint4 xv[kRunVec], yv[kRunVec];
#pragma unroll
    for (int q = 0; q < kRunVec; ++q) {
        const int v = v0 + q;
        const bool in = v < v_end;
        xv[q] = in ? __ldcg(tv + v) : make_uint4(0, 0, 0, 0);
        yv[q] = in && resid ? __ldcg(dv + v) : make_uint4(0, 0, 0, 0);
    }
    float vs[kRunVec];
    float ls = 0.f;
#pragma unroll
    for (int q = 0; q < kRunVec; ++q) {
        float w[VE];
        weights(xv[q], yv[q], w);
        vs[q] = v0 + q < v_end ? pair_sum<VE>(w) : 0.f;
        ls += vs[q];
    }
    const F2 incl = warp_scan_incl(f2(ls), lane);
    const F2 prev = f2_shfl_up(incl, 1);
    const F2 excl = lane > 0 ? prev : f2(0.f);
    const unsigned hit = __ballot_sync(0xffffffffu, ls > 0.f && f2_gt(incl, target));
    const unsigned pos = __ballot_sync(0xffffffffu, ls > 0.f);
    const int lsel = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
    if (lsel < 0) return y0;  // a slot without weight (not drawn in practice)
    int pick = -1;
    if (lane == lsel) {
        float run = 0.f, run_at = 0.f;
        int qsel = -1, qlast = -1;
#pragma unroll
        for (int q = 0; q < kRunVec; ++q) {
            if (qsel < 0 && vs[q] > 0.f) {
                qlast = q;
                run_at = run;
                if (f2_gt(excl + f2(run + vs[q]), target)) qsel = q;
            }
            run += vs[q];
        }
        if (qsel < 0) qsel = qlast;
        int lastpos = -1;
#pragma unroll
        for (int q = 0; q < kRunVec; ++q) {
            if (q != qsel) continue;
            float w[VE];
            weights(xv[q], yv[q], w);
            float re = run_at;
#pragma unroll
            for (int e = 0; e < VE; ++e) {
                re += w[e];
                if (pick < 0 && w[e] > 0.f) {
                    lastpos = (v0 + q) * VE + e;
                    if (f2_gt(excl + f2(re), target)) pick = (v0 + q) * VE + e;
                }
            }
        }
        if (pick < 0) pick = lastpos >= 0 ? lastpos : v0 * VE;
    }
    return __shfl_sync(0xffffffffu, pick, lsel);
}

// The token inside sampling block `blk` of packed target row r, given the
// block's per-warp slot masses sm_w (w < wpb, in every lane): the slot whose
// running mass crosses u_tok times the block mass, then the id inside it.
template <typename T>
__device__ int block_pick(const VerifyArgs &a, const DecideState &st, int b, int r, int blk,
                          const float (&slot_mass)[kCW], int wpb, int tpw, int lane) {
    F2 total = f2(0.f);
#pragma unroll
    for (int w = 0; w < kCW; ++w)
        if (w < wpb) total = total + f2(slot_mass[w]);
    const F2 target = f2_scale(total, st.u_tok);
    F2 cum = f2(0.f), before = f2(0.f);
    int wsel = -1, wlast = 0;
#pragma unroll
    for (int w = 0; w < kCW; ++w) {
        if (w >= wpb || wsel >= 0) continue;
        if (slot_mass[w] > 0.f) {
            wlast = w;
            if (f2_gt(cum + f2(slot_mass[w]), target)) {
                wsel = w;
                before = cum;
            }
        }
        cum = cum + f2(slot_mass[w]);
    }
    if (wsel < 0) {
        wsel = wlast;
        before = f2(0.f);
#pragma unroll
        for (int w = 0; w < kCW; ++w)
            if (w < wsel) before = before + f2(slot_mass[w]);
    }
    return slot_pick<T>(a, st, b, r, blk * kSampleBlock + wsel * tpw, tpw, target - before, lane);
}

// (max, sum) of p over sampling block i of request b's bonus row, from the
// per-warp slots.
__device__ __forceinline__ float2 bonus_block(const VerifyArgs &a, int b, int i, int wpb,
                                              float scale) {
    const float2 *sl = a.blkrec + (size_t(b) * a.nblk + i) * kCW;
    float2 x[kCW];
#pragma unroll
    for (int w = 0; w < kCW; ++w) x[w] = w < wpb ? __ldcg(sl + w) : make_float2(-INFINITY, 0.f);
    float m = -INFINITY, s = 0.f;
#pragma unroll
    for (int w = 0; w < kCW; ++w) ms_combine(m, s, x[w].x, x[w].y, scale);
    return make_float2(m, s);
}

// A sampling draw's inputs, from the bonus row's slots or the residual
// masses: the slot masses of blocks lane and lane + 32 in every lane
// (blocks from 64 on are read again by slot_mass_at), the drawn row's
// state, the kind of slot record, and what the commit needs.  Both draws
// then share one tail (draw_tail), inlined once in the decider: its code is
// cold beside the consumers' loop, and less of it makes the chain shorter.
struct DrawPrep {
    DecideState st;
    float m[2][kCW];  // slot masses of blocks lane, lane + 32 (0 past the row)
    float M;          // bonus: the reference of the slot masses
    int kind;         // 0: bonus-row slots, 1: residual masses, 2: p masses
    int r;            // packed target row drawn from
    int acc;          // committed drafts
    Drafts dr;
};

// Mass of slot w of block i of request b, read from the workspace (kind as
// in DrawPrep).
__device__ __forceinline__ float slot_mass_at(const VerifyArgs &a, int kind, int b, int i, int w,
                                              float M) {
    const size_t o = (size_t(b) * a.nblk + i) * kCW + w;
    if (kind == 0) {
        const float2 x = __ldcg(a.blkrec + o);
        return x.y > 0.f ? x.y * exp2_approx((x.x - M) * a.scale) : 0.f;
    }
    const float2 x = __ldcg(a.zrec + o);
    return kind == 1 ? x.x : x.y;
}

// The bonus draw of request b, every draft accepted: from p of row L_b
// (sampling; block and slot masses from the row's per-warp slots), or the
// argmax of row L_b (greedy; from its chunk records).  Sampling prepares
// the draw and returns true; greedy commits and returns false.
template <typename T>
__device__ bool prep_bonus(const VerifyArgs &a, const StreamShape &sh, int b, DrawPrep &p,
                           int wpb, int lane) {
    const int Lb = verify_len(a, b), r = a.row_off[b] + Lb;
    p.dr = load_drafts(a, b, lane);
    if (a.greedy) {
        float v = -INFINITY;
        int id = INT_MAX;
        const float4 *rec = a.rowrec + size_t(r) * a.grp_stride;
        for (int g = lane; g < sh.gprbQ; g += 32) {
            const float4 x = __ldcg(rec + g);
            am_combine(v, id, x.x, __float_as_int(x.y));
        }
        warp_am_reduce(v, id);
        finish_request(a, b, Lb, id, p.dr, lane);
        return false;
    }
    const float scale = a.scale;
    float2 sl[2][kCW];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int i = q * 32 + lane;
        const float2 *x = a.blkrec + (size_t(b) * a.nblk + (i < a.nblk ? i : 0)) * kCW;
#pragma unroll
        for (int w = 0; w < kCW; ++w)
            sl[q][w] = i < a.nblk && w < wpb ? __ldcg(x + w) : make_float2(-INFINITY, 0.f);
    }
    float u, ub, ut;
    step_uniforms(a.seed, b, Lb, u, ub, ut);
    float mb = -INFINITY;
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int w = 0; w < kCW; ++w)
            if (sl[q][w].y > 0.f) mb = fmaxf(mb, sl[q][w].x);
    for (int i = 64 + lane; i < a.nblk; i += 32) {
        const float2 x = bonus_block(a, b, i, wpb, scale);
        if (x.y > 0.f) mb = fmaxf(mb, x.x);
    }
    const float M = warp_max(mb);
    // slot mass in the units of 2^((z - M) s)
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int w = 0; w < kCW; ++w)
            p.m[q][w] = sl[q][w].y > 0.f ? sl[q][w].y * exp2_approx((sl[q][w].x - M) * scale) : 0.f;
    p.M = M;
    p.kind = 0;
    p.r = r;
    p.acc = Lb;
    p.st.a = Lb;
    p.st.mode = D_BONUS;
    p.st.Mp = M;
    p.st.Sp = 1.f;
    p.st.Mq = 0.f;
    p.st.Sq = 1.f;
    p.st.u_blk = ub;
    p.st.u_tok = ut;
    return true;
}

// Request b's decision rows (k < L_b) are all in: accept tests and outputs
// of the draft rows.  A rejection starts the residual draw (sampling) or
// emits the row's argmax (greedy) and marks the request so its bonus row is
// not streamed; with every draft accepted the bonus draw runs once the bonus
// row is in too (join counter: whichever comes second runs it).  Loads that
// do not depend on one another are issued together: a decision runs while
// the streaming keeps L2 busy, and each dependent round trip costs
// microseconds.
template <typename T>
__device__ bool decide_request(const VerifyArgs &a, const StreamShape &sh, int b, int wpb,
                               int epoch, int lane) {
    // Round 1: lengths, offsets and draft tokens.
    const int Lb = verify_len(a, b), r0 = a.row_off[b], d0 = a.draft_off[b];
    // Committed window: L_b, or in the cap-accept audit the scheduled W_b
    // clamped to [0, L_b] (the full block is verified, the window committed).
    const int W = a.commit_len ? min(max(__ldcg(a.commit_len + b), 0), Lb) : Lb;
    const Drafts dr = load_drafts(a, b, lane);
    const float scale = a.scale;
    int ab = Lb;                                   // first rejected draft (L_b: none)
    // Normalisers and uniforms of the row the emitted token is drawn from:
    // min(a_b, W) -- row a_b after a rejection inside the window, row W when
    // the window ends inside the accepted run.
    float Mp = 0.f, Sp = 0.f, Mq = 0.f, Sq = 0.f;
    float ub = 0.f, ut = 0.f;
    int g_tok = 0;
    // Round 2, one lane per row k (two rounds when gamma > 32): the row's
    // chunk records and its gathered z values.
    for (int base = 0; base < Lb; base += 32) {
        const int k = base + lane;
        const bool live = k < Lb;
        const int r = r0 + k;
        const int nrec = r < sh.nA ? 1 : r < sh.nB ? sh.gprb : a.nc;
        const float4 *rec = a.rowrec + size_t(live ? r : r0) * a.grp_stride;
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            x[u] = live && u < nrec ? __ldcg(rec + u) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float2 z = !a.greedy && live ? __ldcg(a.gath + r) : make_float2(0.f, 0.f);
        float u = 1.f, u1 = 0.f, u2 = 0.f;
        if (!a.greedy && live) step_uniforms(a.seed, b, k, u, u1, u2);
        float4 rr = a.greedy ? make_float4(-INFINITY, __int_as_float(INT_MAX), 0.f, 0.f)
                             : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        if (live) {
            for (int i0 = 0; i0 < nrec; i0 += 4) {
                if (i0 > 0) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        if (i0 + v < nrec) x[v] = __ldcg(rec + i0 + v);
                }
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    if (i0 + v >= nrec) continue;
                    if (a.greedy) {
                        int bi = __float_as_int(rr.y);
                        am_combine(rr.x, bi, x[v].x, __float_as_int(x[v].y));
                        rr.y = __int_as_float(bi);
                    } else {
                        ms_combine(rr.x, rr.y, x[v].x, x[v].y, scale);
                        ms_combine(rr.z, rr.w, x[v].z, x[v].w, scale);
                    }
                }
            }
        }
        bool accept = false;
        if (live) {
            const int dt = base == 0 ? dr.t[0] : dr.t[1];
            if (a.greedy) {
                accept = dt == __float_as_int(rr.y);
                a.p_tok[d0 + k] = 0.f;
                a.q_tok[d0 + k] = 0.f;
            } else {
                float p = 0.f, q = 0.f, ratio = 0.f;
                if (dt >= 0 && dt < a.V) {
                    p = exp2_approx((z.x - rr.x) * scale) / rr.y;
                    q = exp2_approx((z.y - rr.z) * scale) / rr.w;
                    ratio = q > 0.f ? fminf(1.f, p / q) : 1.f;
                }
                accept = u < ratio;
                a.p_tok[d0 + k] = p;
                a.q_tok[d0 + k] = q;
            }
        }
        const unsigned acc = __ballot_sync(0xffffffffu, live && accept);
        const unsigned rows = __ballot_sync(0xffffffffu, live);
        const unsigned rej = rows & ~acc;
        if (ab == Lb && rej) ab = base + __ffs(rej) - 1;
        const int src = min(ab, W) - base;
        const int sl_ = src >= 0 && src < 32 ? src : 0;
        const float m1 = __shfl_sync(0xffffffffu, rr.x, sl_), s1 = __shfl_sync(0xffffffffu, rr.y, sl_);
        const float m2 = __shfl_sync(0xffffffffu, rr.z, sl_), s2 = __shfl_sync(0xffffffffu, rr.w, sl_);
        const float v1 = __shfl_sync(0xffffffffu, u1, sl_), v2 = __shfl_sync(0xffffffffu, u2, sl_);
        if (src >= 0 && src < 32) {
            Mp = m1;
            Sp = s1;
            Mq = m2;
            Sq = s2;
            ub = v1;
            ut = v2;
            g_tok = __float_as_int(s1);  // greedy: the row's argmax
        }
    }
    const int acc = min(ab, W);  // committed drafts
    if (lane == 0 && a.accept_full) a.accept_full[b] = ab;
    if (lane == 0 && a.audit_totals) {
        atomicAdd(&a.q_ctr[Q_AFULL], ab);
        atomicAdd(&a.q_ctr[Q_ACOMMIT], acc);
    }
    if (acc < Lb) {
        // A rejection inside the window (residual draw at row a_b), or a
        // window that ends inside the accepted run (draw from p at row W,
        // what compact's bonus draw would be).  The bonus row is not needed.
        if (lane == 0) st_relaxed(&a.rejflag[b], epoch);  // phase Q skips the bonus row
        if (a.greedy) {
            finish_request(a, b, acc, g_tok, dr, lane);
            return false;
        }
        DecideState st;
        st.a = acc;
        st.mode = ab < W ? D_RESID : D_FALLBACK;
        st.Mp = Mp;
        st.Sp = Sp;
        st.Mq = Mq;
        st.Sq = Sq;
        st.u_blk = ub;
        st.u_tok = ut;
        if (lane == 0) {
            a.dstate[b] = st;
            push_resid_jobs(a, b, epoch);
        }
        return false;
    }
    // Every draft accepted: the bonus draw (true), if the bonus row is in
    // already.
    int go = 0;
    if (lane == 0) {
        fence_acq_rel_gpu();
        go = atomicAdd(&a.join[b], 1) == 1;
    }
    const bool run = __shfl_sync(0xffffffffu, go, 0) != 0;
    if (run) fence_acq_rel_gpu();
    return run;
}

// Every residual slot of request b is in: the residual draw at packed row
// r from the masses, or a draw from p of the same row when there is no
// residual mass (or the window ends inside the accepted run).
template <typename T>
__device__ void prep_residual(const VerifyArgs &a, int b, int r, DecideState st, DrawPrep &p,
                              int wpb, int lane) {
    // One round of independent loads: drafts, masses.
    p.dr = load_drafts(a, b, lane);
    const float2 *z = a.zrec + size_t(b) * a.nblk * kCW;
    float2 sl[2][kCW];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int i = q * 32 + lane;
#pragma unroll
        for (int w = 0; w < kCW; ++w)
            sl[q][w] = i < a.nblk && w < wpb ? __ldcg(z + size_t(i) * kCW + w) : make_float2(0.f, 0.f);
    }
    // Residual mass anywhere in the row (masses are sums of non-negative
    // terms: their total is positive exactly when one of them is).
    bool pos = false;
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int w = 0; w < kCW; ++w) pos |= sl[q][w].x > 0.f;
    for (int i = 64 + lane; i < a.nblk; i += 32)
        for (int w = 0; w < wpb; ++w) pos |= __ldcg(z + size_t(i) * kCW + w).x > 0.f;
    const bool residual = st.mode == D_RESID && __any_sync(0xffffffffu, pos);
    if (!residual) {
        st.mode = D_FALLBACK;
        st.Sp = 1.f;
    }
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int w = 0; w < kCW; ++w) p.m[q][w] = residual ? sl[q][w].x : sl[q][w].y;
    p.M = 0.f;
    p.kind = residual ? 1 : 2;
    p.r = r;
    p.acc = st.a;
    p.st = st;
}

// The end of every sampling draw of request b: the block by u' from the
// block masses, the slot inside it, then the id by u''; the commit.
template <typename T>
__device__ void draw_tail(const VerifyArgs &a, int b, const DrawPrep &p, int wpb, int lane) {
    F2 bm[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) bm[q] = sum8_f2(p.m[q]);
    // block i's mass, evaluated by the lane owning it
    auto mass = [&](int i) {
        if (i < 64) return i < 32 ? bm[0] : bm[1];
        F2 m = f2(0.f);
        for (int w = 0; w < wpb; ++w) m = m + f2(slot_mass_at(a, p.kind, b, i, w, p.M));
        return m;
    };
    const int blk = choose_block(a.nblk, p.st.u_blk, mass, lane);
    float slot_mass[kCW];
    const int q = blk >> 5, owner = blk & 31;
#pragma unroll
    for (int w = 0; w < kCW; ++w) {
        float m = 0.f;
        if (q < 2) m = __shfl_sync(0xffffffffu, q == 0 ? p.m[0][w] : p.m[1][w], owner);
        else if (w < wpb) m = slot_mass_at(a, p.kind, b, blk, w, p.M);
        slot_mass[w] = w < wpb ? m : 0.f;
    }
    const int token = block_pick<T>(a, p.st, b, p.r, blk, slot_mass, wpb, kSampleBlock / wpb, lane);
    finish_request(a, b, p.acc, token, p.dr, lane);
}

// ---------------------------------------------------------------------------
// consumers
// ---------------------------------------------------------------------------
template <typename T>
__device__ void consumer(const VerifyArgs &a, VSmem &sm, const uint8_t *ring,
                         const StreamShape &sh, int warp, int lane, int epoch) {
    constexpr int VE = Vec<T>::kElems;
    const float scale = a.scale;
    const int tpw = a.chunk_elems / kCW;  // tokens per warp in a tile
    const int vpw = tpw / VE;             // vectors per warp in a tile
    // Row accumulators of pair rows (sampling) / of every row (greedy),
    // carried across the tiles of a chunk.
    float mr[2] = {-INFINITY, -INFINITY}, sr[2] = {0.f, 0.f};  // (p, q) of a pair row
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int fill = 0;; ++fill) {
        const int s = fill % kStages, n = fill / kStages;
        if (!mbar_wait_backoff(&sm.full[s], n & 1, a.wait_ns)) {
            if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
            return;
        }
        const TaskInfo t = sm.task[s];
        if (t.type == T_EXIT) return;
        const uint4 *tv = reinterpret_cast<const uint4 *>(ring + s * kStageBytes);
        const uint4 *dv = tv + kChunkBytes / 16;
        const int nvec = t.bytes / 16;
        const int v0 = min(nvec, warp * vpw), v1 = min(nvec, v0 + vpw);

        if (t.type == T_STREAM) {
            if (a.greedy) {
                for (int h = 0; h < (t.bytes2 > 0 ? 2 : 1); ++h) {
                    const uint4 *xv = h ? dv : tv;
                    const int nv = (h ? t.bytes2 : t.bytes) / 16;
                    const int va = min(nv, warp * vpw), vb = min(nv, va + vpw);
                    const int yb = t.y0 + h * a.chunk_elems;
                    for (int v = va + lane; v < vb; v += 32) {
                        float z[VE];
                        Vec<T>::unpack(xv[v], z);
#pragma unroll
                        for (int e = 0; e < VE; ++e)
                            if (z[e] > bv) {
                                bv = z[e];
                                bi = yb + v * VE + e;
                            }
                    }
                }
            } else if (t.pair) {
                const uint4 *const rows[2] = {tv, dv};
                tile_fold<T, 2>(mr, sr, rows, v0, v1, lane, scale);
                if (lane == 0) {
                    const int lo = t.y0 + v0 * VE, hi = t.y0 + v1 * VE;
                    if (t.d >= lo && t.d < hi)
                        a.gath[t.r] = make_float2(Vec<T>::load1(tv, t.d - t.y0),
                                                  Vec<T>::load1(dv, t.d - t.y0));
                }
            } else {
                // Bonus row: one (max, sum) slot per tile and warp.
                for (int h = 0; h < (t.bytes2 > 0 ? 2 : 1); ++h) {
                    const uint4 *xv = h ? dv : tv;
                    const int nv = (h ? t.bytes2 : t.bytes) / 16;
                    const int va = min(nv, warp * vpw), vb = min(nv, va + vpw);
                    float bm[1] = {-INFINITY}, bs[1] = {0.f};
                    const uint4 *const rows[1] = {xv};
                    tile_fold<T, 1>(bm, bs, rows, va, vb, lane, scale);
                    warp_ms_reduce(bm[0], bs[0], scale);
                    const int y = t.y0 + h * a.chunk_elems + warp * tpw;
                    const int blk = y / kSampleBlock;
                    if (lane == 0 && blk < a.nblk)
                        a.blkrec[(size_t(t.b) * a.nblk + blk) * kCW + (y % kSampleBlock) / tpw] =
                            make_float2(bm[0], bs[0]);
                }
            }
            if (t.flush && (a.greedy || t.pair)) {
                // End of the chunk: the eight warp partials become one record.
                if (a.greedy) {
                    warp_am_reduce(bv, bi);
                    if (lane == 0) sm.part[s][warp] = make_float4(bv, __int_as_float(bi), 0.f, 0.f);
                } else {
                    warp_ms_reduce(mr[0], sr[0], scale);
                    warp_ms_reduce(mr[1], sr[1], scale);
                    if (lane == 0) sm.part[s][warp] = make_float4(mr[0], sr[0], mr[1], sr[1]);
                }
                mr[0] = mr[1] = bv = -INFINITY;
                sr[0] = sr[1] = 0.f;
                bi = INT_MAX;
                int last = 0;
                if (lane == 0) {
                    __threadfence_block();
                    last = atomicAdd(&sm.done[s], 1) == kCW - 1;
                }
                if (__shfl_sync(0xffffffffu, last, 0)) {
                    __threadfence_block();
                    float4 x = lane < kCW ? sm.part[s][lane]
                                          : (a.greedy ? make_float4(-INFINITY, __int_as_float(INT_MAX), 0.f, 0.f)
                                                      : make_float4(-INFINITY, 0.f, -INFINITY, 0.f));
                    if (a.greedy) {
                        int xi = __float_as_int(x.y);
                        warp_am_reduce(x.x, xi);
                        x.y = __int_as_float(xi);
                    } else {
                        warp_ms_reduce(x.x, x.y, scale);
                        warp_ms_reduce(x.z, x.w, scale);
                    }
                    if (lane == 0) {
                        sm.done[s] = 0;
                        a.rowrec[size_t(t.r) * a.grp_stride + t.g] = x;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
        } else {
            // Residual tile: this warp's share of the residual and p masses.
            const float iSp = 1.f / t.Sp, iSq = 1.f / t.Sq;
            float zr = 0.f, zp = 0.f;
            for (int v = v0 + lane; v < v1; v += 32) {
                float x[VE], y[VE];
                Vec<T>::unpack(tv[v], x);
                Vec<T>::unpack(dv[v], y);
#pragma unroll
                for (int e = 0; e < VE; ++e) {
                    const float pw = exp2_approx((x[e] - t.Mp) * scale);
                    zp += pw;
                    zr += fmaxf(0.f, pw * iSp - exp2_approx((y[e] - t.Mq) * scale) * iSq);
                }
            }
            const F2 dr = warp_sum_f2(f2(zr)), dp = warp_sum_f2(f2(zp));
            // The masses are written before the stage is released: the
            // producer books the tile (and publishes it) once all eight warps
            // have released it.
            const int y = t.y0 + warp * tpw;
            const int blk = y / kSampleBlock;
            if (lane == 0 && blk < a.nblk)
                a.zrec[(size_t(t.b) * a.nblk + blk) * kCW + (y % kSampleBlock) / tpw] =
                    make_float2(dr.hi + dr.lo, dp.hi + dp.lo);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
        }
    }
}

// ---------------------------------------------------------------------------
// decider: warp kCW + 1 serves the decide queue, and between jobs feeds its
// producer's residual-tile mailbox
// ---------------------------------------------------------------------------
template <typename T>
__device__ void decider(const VerifyArgs &a, VSmem &sm, const StreamShape &sh, int epoch,
                        int lane) {
    static_assert(QA_HEAD == 0 && QA_TAIL == 1 && Q_FINISHED == 2, "one vector load");
    const int wpb = kSampleBlock / (a.chunk_elems / kCW);
    int pending = -1;  // decide-queue index
    int rclaim = -1;   // residual-queue index claimed for this CTA's producer
    for (;;) {
        int b = -1;
        if (lane == 0) {
            if (pending < 0) pending = atomicAdd(&a.q_ctr[QB_HEAD], 1);
            const uint64_t t0 = global_timer_ns();
            unsigned ns = 32;
            for (;;) {
                if (rclaim >= 0) {
                    // A claimed residual tile goes out before anything else:
                    // its job was queued when it was claimed, so its ready
                    // word follows within the pusher's few stores.
                    if (ld_acquire(&a.q_ready[rclaim]) == epoch) {
                        mbox_put(sm, resid_task(a, __ldcg(a.q_job + rclaim)));
                        rclaim = -1;
                        ns = 32;
                        continue;
                    }
                } else {
                    if (pending < a.qbcap && ld_acquire(&a.qb_ready[pending]) == epoch) {
                        b = __ldcg(a.qb_job + pending);
                        pending = -1;
                        break;
                    }
                    const int4 q = ld_acquire_ctr4(a.q_ctr);
                    if (q.z >= a.B) break;
                    // The mailbox is empty and a residual tile is queued:
                    // claim its index, never one past the tail, so that a
                    // claim is always served at once.
                    if (q.x < q.y && q.x < a.qcap && mbox_empty(sm) &&
                        atomicCAS(&a.q_ctr[QA_HEAD], q.x, q.x + 1) == q.x)
                        rclaim = q.x;
                    if (rclaim >= 0) continue;
                }
                if (global_timer_ns() - t0 > a.wait_ns) {
                    atomicOr(a.status, kStatusQueueTimeout);
                    break;
                }
                __nanosleep(ns);
                ns = min(ns * 2, 256u);
            }
        }
        b = __shfl_sync(0xffffffffu, b, 0);
        if (b < 0) return;  // the ready word was read with acquire: no fence needed
        // Every sampling draw goes through the one draw_tail below.
        DrawPrep dp;
        bool draw = false, bonus = false;
        if (b & kFinishResidual) {
            b &= ~kFinishResidual;
            const DecideState st = load_state(a, b);
            prep_residual<T>(a, b, a.row_off[b] + st.a, st, dp, wpb, lane);
            draw = true;
        } else if (b & kBonusDraw) {
            b &= ~kBonusDraw;
            bonus = true;
        } else {
            bonus = decide_request<T>(a, sh, b, wpb, epoch, lane);
        }
        if (bonus) draw = prep_bonus<T>(a, sh, b, dp, wpb, lane);
        if (draw) draw_tail<T>(a, b, dp, wpb, lane);
    }
}

template <typename T>
__global__ void __launch_bounds__(kVerifyThreads, 2) verify_kernel(const VerifyArgs a) {
    extern __shared__ __align__(1024) uint8_t ring[];
    __shared__ VSmem sm;
    // Launched as a programmatic dependent: wait until the grid before it has
    // completed and its writes (offsets, packed rows) are visible.  Without
    // such a grid this returns at once.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int epoch = a.q_ctr[Q_EPOCH] + 1;
    // The producer's first row ids go out with the packed total (the row-id
    // arrays hold the batch's capacity): one round trip less before the
    // CTA's first copy.
    const bool prod = warp == kCW && lane == 0;
    const int pre_b = prod && int(blockIdx.x) < a.B * (a.gamma + 1) ? a.row_req[blockIdx.x] : -1;
    const int pre_k = prod && int(blockIdx.x) < a.B * (a.gamma + 1) ? a.row_k[blockIdx.x] : 0;
    const StreamShape sh = stream_shape(a);
    if (tid < kStages) {
        mbar_init(&sm.full[tid], 1);
        mbar_init(&sm.empty[tid], kCW);
        sm.done[tid] = 0;
    }
    if (tid == 0) sm.mbox_full = 0;
    if (tid == 0) fence_barrier_init();
    __syncthreads();
    if (warp == kCW) {
        if (lane == 0) producer(a, sm, ring, sh, epoch, pre_b, pre_k);
    } else if (warp == kCW + 1) {
        decider<T>(a, sm, sh, epoch, lane);
    } else {
        consumer<T>(a, sm, ring, sh, warp, lane, epoch);
    }
    __syncthreads();
    __shared__ int s_last;
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(&a.q_ctr[Q_EXITED], 1) == int(gridDim.x) - 1;
    }
    __syncthreads();
    if (s_last) {
        // Every CTA is done.  Bonus-row counts of requests that rejected can
        // arrive after the request finished, so these reset here.
        for (int b = tid; b < a.B; b += kVerifyThreads) {
            a.bon_cnt[b] = 0;
            a.join[b] = 0;
        }
        if (tid == 0) {
            // Reset the queues for the next launch.
            a.q_ctr[QA_HEAD] = 0;
            a.q_ctr[QA_TAIL] = 0;
            a.q_ctr[QB_HEAD] = 0;
            a.q_ctr[QB_TAIL] = 0;
            a.q_ctr[Q_FINISHED] = 0;
            a.q_ctr[Q_CHUNK] = 0;
            a.q_ctr[Q_EXITED] = 0;
            a.q_ctr[Q_EPOCH] = epoch;
            if (a.audit_totals) {
                a.audit_totals[0] = atomicExch(&a.q_ctr[Q_AFULL], 0);
                a.audit_totals[1] = atomicExch(&a.q_ctr[Q_ACOMMIT], 0);
            }
        }
        __threadfence();
    }
}

// ---------------------------------------------------------------------------
// tail kernel (sampling): residual rows and draws
// ---------------------------------------------------------------------------
// After the small-batch verify: the second pass over the row of each
// rejection it listed (the row's residual masses) and the residual draw.
// One CTA alone needs ~25 us for a 300 KB row pair (a few dozen KB in flight
// per round trip); here each row is cut into parts over the whole GPU.
constexpr int kTailThreads = kCW * 32;
constexpr int kTailRun = kChunkBytes / 16 / kCW / 32;  // 16-byte vectors a lane sums per slot
constexpr int kTailParts = 4;                          // units per listed row
constexpr int kTailBatch = 2;                          // tiles whose loads are in flight together

// Tiles [t0, t1) of a listed row -- target row r and draft row (b, a_b):
// warp w sums max(0, p - q) and p over slot w of each tile, with the lanes
// and order the stream kernel's consumers use for a slot, and writes the
// slot's masses.
template <typename T>
__device__ void residual_part(const VerifyArgs &a, const DecideState &st, int b, int r, int t0,
                              int t1, int warp, int lane) {
    constexpr int VE = Vec<T>::kElems;
    const int tpw = a.chunk_elems / kCW, vpw = tpw / VE;
    const float scale = a.scale, iSp = 1.f / st.Sp, iSq = 1.f / st.Sq;
    const char *trow = static_cast<const char *>(a.target_logits) + size_t(r) * a.row_bytes;
    const char *drow = static_cast<const char *>(a.draft_logits) +
                       (size_t(b) * a.gamma + st.a) * size_t(a.row_bytes);
    for (int j0 = t0; j0 < t1; j0 += kTailBatch) {
        uint4 xs[kTailBatch][kTailRun], ys[kTailBatch][kTailRun];
        int v0[kTailBatch], v1[kTailBatch];
#pragma unroll
        for (int h = 0; h < kTailBatch; ++h) {
            const int j = j0 + h;
            const int nvec = j < t1 ? min(kChunkBytes, a.row_bytes - j * kChunkBytes) / 16 : 0;
            v0[h] = min(nvec, warp * vpw);
            v1[h] = min(nvec, v0[h] + vpw);
            const uint4 *tv = reinterpret_cast<const uint4 *>(trow + size_t(j) * kChunkBytes);
            const uint4 *dv = reinterpret_cast<const uint4 *>(drow + size_t(j) * kChunkBytes);
#pragma unroll
            for (int q = 0; q < kTailRun; ++q) {
                const int v = v0[h] + lane + 32 * q;
                xs[h][q] = v < v1[h] ? __ldcg(tv + v) : make_uint4(0, 0, 0, 0);
                ys[h][q] = v < v1[h] ? __ldcg(dv + v) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int h = 0; h < kTailBatch; ++h) {
            const int j = j0 + h;
            if (j >= t1) break;
            float zr = 0.f, zp = 0.f;
#pragma unroll
            for (int q = 0; q < kTailRun; ++q) {
                if (v0[h] + lane + 32 * q >= v1[h]) continue;
                float x[VE], y[VE];
                Vec<T>::unpack(xs[h][q], x);
                Vec<T>::unpack(ys[h][q], y);
#pragma unroll
                for (int e = 0; e < VE; ++e) {
                    const float pw = exp2_approx((x[e] - st.Mp) * scale);
                    zp += pw;
                    zr += fmaxf(0.f, pw * iSp - exp2_approx((y[e] - st.Mq) * scale) * iSq);
                }
            }
            const F2 dr = warp_sum_f2(f2(zr)), dp = warp_sum_f2(f2(zp));
            const int y = j * a.chunk_elems + warp * tpw;
            const int blk = y / kSampleBlock;
            if (lane == 0 && blk < a.nblk)
                a.zrec[(size_t(b) * a.nblk + blk) * kCW + (y % kSampleBlock) / tpw] =
                    make_float2(dr.hi + dr.lo, dp.hi + dp.lo);
        }
    }
}

// Units: each listed row in kTailParts parts; the CTA that completes a row
// makes its draw.
template <typename T>
__global__ void __launch_bounds__(kTailThreads) verify_tail_kernel(const VerifyArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ int s_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_rows = min(a.q_ctr[kQSmallList], a.B);
    const int n_res = n_rows * kTailParts;
    const int wpb = kSampleBlock / (a.chunk_elems / kCW);
    const int per = (a.nc + kTailParts - 1) / kTailParts;  // tiles per part
    const int parts = (a.nc + per - 1) / per;               // parts a row has
    for (int u = blockIdx.x; u < n_res; u += gridDim.x) {
        const int i = u / kTailParts, part = u - i * kTailParts;
        if (part >= parts) continue;
        const int2 jb = __ldcg(a.q_job + i);  // (b, r)
        const DecideState st = load_state(a, i);
        residual_part<T>(a, st, jb.x, jb.y, part * per, min(a.nc, (part + 1) * per), warp,
                         lane);
        __syncthreads();
        if (tid == 0) {
            __threadfence();  // every warp's masses (the barrier) before the count
            s_flag = atomicAdd(&a.r1_cnt[jb.x], 1) == parts - 1;
            if (s_flag) __threadfence();  // and every other CTA's, before they are read
        }
        __syncthreads();
        if (s_flag && warp == 0) {
            DrawPrep dp;
            prep_residual<T>(a, jb.x, jb.y, st, dp, wpb, lane);
            draw_tail<T>(a, jb.x, dp, wpb, lane);
        }
    }
    // The last CTA out resets the list for the next launch.
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        s_flag = atomicAdd(&a.q_ctr[kQTailExit], 1) == int(gridDim.x) - 1;
    }
    __syncthreads();
    if (s_flag && tid == 0) {
        a.q_ctr[kQSmallList] = 0;
        a.q_ctr[kQTailExit] = 0;
    }
}

}  // namespace

size_t verify_smem_bytes() { return kSmemBytes; }

int verify_blocks_per_sm(int logit_bf16) {
    cudaError_t e =
        logit_bf16 ? cudaFuncSetAttribute(verify_kernel<uint16_t>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes))
                   : cudaFuncSetAttribute(verify_kernel<float>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
    if (e != cudaSuccess) return -1;
    int n = 0;
    e = logit_bf16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, verify_kernel<uint16_t>,
                                                                   kVerifyThreads, kSmemBytes)
                   : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, verify_kernel<float>,
                                                                   kVerifyThreads, kSmemBytes);
    return e == cudaSuccess ? n : -1;
}

cudaError_t launch_verify(const VerifyArgs &a, int logit_bf16, int grid, cudaStream_t s) {
    // A programmatic dependent of the kernel before it (the score kernel or
    // the compaction): the grid is scheduled while that kernel finishes and
    // waits for it at its start (griddepcontrol.wait).  Not cooperative: one
    // CTA per resident slot, so every CTA runs at once; the stream chunks
    // after each CTA's first, the residual tiles and the decider jobs are
    // claimed by running CTAs, and every wait is bounded.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kVerifyThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (logit_bf16) return cudaLaunchKernelEx(&cfg, verify_kernel<uint16_t>, a);
    return cudaLaunchKernelEx(&cfg, verify_kernel<float>, a);
}

int verify_tail_blocks_per_sm(int logit_bf16) {
    int n = 0;
    const cudaError_t e =
        logit_bf16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, verify_tail_kernel<uint16_t>,
                                                                   kTailThreads, 0)
                   : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, verify_tail_kernel<float>,
                                                                   kTailThreads, 0);
    return e == cudaSuccess ? n : -1;
}

cudaError_t launch_verify_tail(const VerifyArgs &a, int logit_bf16, int grid, cudaStream_t s) {
    // A programmatic dependent of the small-batch verify: its CTAs take the
    // slots that grid's CTAs leave, and wait for it to complete.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTailThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (logit_bf16) return cudaLaunchKernelEx(&cfg, verify_tail_kernel<uint16_t>, a);
    return cudaLaunchKernelEx(&cfg, verify_tail_kernel<float>, a);
}

}  // namespace dspark
