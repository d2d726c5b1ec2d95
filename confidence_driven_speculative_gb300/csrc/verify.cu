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
// and every kept draft row (sum L) is read at most once, V logits each; a
// rejected request's row pair is read once more for its residual.
//
// One persistent cooperative grid, a few CTAs per SM, in three phases
// separated by grid barriers:
//
//  1. Stream.  Each CTA is a producer warp, 8 consumer warps and a decider
//     warp.  The producer fills a 3-stage shared-memory ring with 1-D bulk
//     TMA copies (cp.async.bulk) completing on "full" mbarriers with byte
//     counts; each consumer warp releases a stage on its "empty" mbarrier as
//     soon as it has read it.  Work is a sequence of chunks handed out by an
//     atomic counter: first the decision rows (target row k with draft row
//     (b, k) in sampling, k < L_b) in draft order, a few 16 KB tiles per
//     chunk, so a request's rows are spread over many CTAs; then each
//     request's bonus row (k = L_b), skipping requests already known to
//     reject (the method never reads past the first rejection).  A consumer
//     warp owns one eighth of every tile: online (max, sum of
//     2^(z log2(e)/Tm - max)) accumulators for p and q (greedy: max and
//     lowest argmax), reduced once per chunk into a record slot of the row;
//     a bonus row keeps one (max, sum) slot per tile and warp -- the block
//     masses of its draw.  The warp that completes a chunk counts it per
//     request with a device atomic; the CTA whose count completes a request
//     decides it in its decider warp: accept tests, p(d), q(d), a_b, and a
//     rejection marks the request so its bonus row is skipped.
//  2. Residual.  The normalised residual max(0, p - q) of a rejected row
//     pair needs that row's normalisers, known only now.  The tiles of every
//     rejected row pair are spread over the grid and streamed again through
//     the rings (partly still in L2); each warp writes the residual and p
//     masses of its slot.
//  3. Draw.  Every warp of the grid takes requests in turn and makes the
//     draw: the bonus token from p at row L_b (every draft accepted), or the
//     residual token at row a_b.  Draws are two-level: a 4096-id block by mass
//     (u'), then an id inside it (u''); in-block running sums are fp32 over
//     short lane runs combined in two-float (TwoSum) arithmetic, as exact as
//     fp64 on the fast fp32 pipe.
//
// Every wait is bounded (VerifyArgs::wait_ns) and sets a status bit when it
// gives up; a producer that gave up waits for its own copies in flight before
// it leaves.  Counters reset themselves at the end of the launch.
//
// The cap-accept audit arm ("DFlash to DSpark in SGLang", "The confidence
// scheduler and verify modes") is the same launch with a committed window
// W_b: every draft of the block is tested, the commit is min(a_b, W_b), and a
// window that ends inside the accepted run draws from p at row W_b through
// the residual path (what compact's bonus draw would be).
#include <climits>

#include "dspark_internal.cuh"

namespace dspark {
namespace {

constexpr int kCW = kConsumerWarps;
constexpr int kRing = 3;                      // stages of the shared-memory ring
constexpr int kWarpsPerCta = kVerifyThreads / 32;
constexpr int kStageBytes = 2 * kChunkBytes;  // target tile + draft tile
constexpr size_t kSmemBytes = size_t(kRing) * kStageBytes;
constexpr int kFifo = 64;                     // CTA event FIFO slots (power of two)
constexpr int kJobs = 64;                     // CTA draw queue slots (power of two)

enum : int { T_END = 0, T_STREAM = 1, T_RESID = 2 };
enum : int { D_BONUS = 0, D_RESID = 1, D_FALLBACK = 2 };
// Draw still to make for a request after phase 1 (act[b]).
enum : int { A_NONE = 0, A_RESID = 1, A_BONUS = 2 };
// q_ctr words: stream-chunk counter, grid barrier count and generation,
// launch epoch, exited CTAs, rejected requests, audit sums.
enum : int { Q_CHUNK = 0, Q_BAR = 1, Q_BARGEN = 2, Q_EPOCH = 3, Q_EXITED = 4, Q_NREJ = 5,
             Q_AFULL = 8, Q_ACOMMIT = 9 };
// Events the producer posts to its CTA's decider: request b's decision rows
// (EV_P), its bonus row (EV_Q) or its residual tiles (EV_R) are all in.
// Encoded as kEvMark | type << 24 | L_b << 16 | b (b < 2^16, L_b <= 64).
enum : int { EV_P = 1, EV_Q = 2, EV_R = 3 };
constexpr int kEvMark = 1 << 30;

__device__ __forceinline__ int ev_make(int type, int Lb, int b) {
    return kEvMark | (type << 24) | (Lb << 16) | b;
}

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
    int mode;   // residual tile: D_RESID (residual weights) or D_FALLBACK (p)
    float u_tok;           // bonus row / residual tile: the in-block uniform u'' of the draw
    float Mp, Sp, Mq, Sq;  // residual tile: normalisers of the rejected row pair
};

struct VSmem {
    uint64_t full[kRing], empty[kRing];
    TaskInfo task[kRing];
    // Chunk-end partials and the count of warps past a stage, one set per
    // parity of the stage's use: a warp may reach the next use of the stage
    // before the last warp of this one has counted itself.
    float4 part[kRing][2][kCW];
    int done[kRing][2];
    int fifo[kFifo];       // consumer -> decider events (0: empty slot)
    int fifo_tail;         // next slot a consumer claims
    int fifo_head;         // next slot the decider reads
    int prod_done;         // the producer has booked every unit of the phase
    // Draws waiting for a warp (event codes): the decider queues them; any
    // warp without other work -- the decider between events, the consumers
    // and the producer once their phase's stream is done -- takes them.
    int jobs[kJobs];
    int job_tail;          // next slot the decider fills
    int job_head;          // next slot a warp takes
    int no_more;           // the decider has queued the phase's last draw
};

// Grid-wide shape of the stream work, the same in every thread.  Packed row
// i (0 <= i < sum L + B, request by request: decision rows, then the bonus
// row) is cut into cpr chunks of CT tiles; chunk c is row c / cpr.
struct StreamShape {
    int n_rows;    // packed rows
    int n_dec;     // decision rows (sum L)
    int CT;        // tiles per decision chunk
    int cpr;       // chunks per decision row
    int CTQ;       // tiles per bonus chunk
    int cprQ;      // chunks per bonus row
    int nP;        // decision chunks
    int n_chunks;  // decision and bonus chunks
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

__device__ __forceinline__ int ld_vol(const int *p) { return *reinterpret_cast<const volatile int *>(p); }
__device__ __forceinline__ void st_vol(int *p, int v) { *reinterpret_cast<volatile int *>(p) = v; }

// The uniforms (u, u', u'') of draft position k of request b, out of line so
// that decisions and draws share one copy of the generator's code.
__device__ __noinline__ float3 uniforms_of(uint64_t seed, int b, int k) {
    float3 r;
    step_uniforms(seed, b, k, r.x, r.y, r.z);
    return r;
}

__device__ __forceinline__ int verify_len(const VerifyArgs &a, int b) {
    return min(max(a.L[b], 0), a.gamma);
}

__device__ __forceinline__ StreamShape stream_shape(const VerifyArgs &a) {
    StreamShape sh;
    const int cap = a.B * (a.gamma + 1);
    // packed rows and drafts as written by the score and compaction kernels,
    // never more than their capacities
    sh.n_rows = min(max(a.row_off[a.B], 0), cap);
    sh.n_dec = min(max(a.draft_off[a.B], 0), a.B * a.gamma);
    if (sh.n_rows < a.B) sh.n_rows = sh.n_dec = 0;  // not the compaction's offsets: no work
    const long long tiles = (long long)sh.n_rows * a.nc;
    const long long g = gridDim.x;
    // a few tiles per chunk when there is plenty of work (fewer chunk
    // records and events); single tiles when there is little, so that every
    // CTA gets some
    sh.CT = tiles >= 16 * g ? 4 : tiles >= 4 * g ? 2 : 1;
    sh.cpr = (a.nc + sh.CT - 1) / sh.CT;
    sh.CTQ = sh.CT;
    sh.cprQ = sh.cpr;
    sh.nP = sh.n_rows * sh.cpr;
    sh.n_chunks = sh.nP;
    return sh;
}

// Largest b in [0, B) with off[b] <= i (off non-decreasing, off[0] = 0):
// the request of decision i.  A 32-way search by the whole warp, two rounds
// of loads for B <= 1024; off is read-only during the launch (__ldg).
// off_b receives off[b].
__device__ int find_request(const int32_t *off, int B, int i, int lane, int &off_b) {
    int lo = 0, hi = B;
    int val = __ldg(off);
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) >> 5;
        const int p = lo + lane * step;
        const int x = p < hi ? __ldg(off + p) : INT_MAX;
        const unsigned m = __ballot_sync(0xffffffffu, lane == 0 || x <= i);
        const int l = 31 - __clz(m);
        val = __shfl_sync(0xffffffffu, x, l);
        lo += l * step;
        hi = min(hi, lo + step);
    }
    off_b = val;
    return lo;
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

// Inclusive warp scan (lane order).
__device__ __forceinline__ F2 warp_scan_incl(F2 v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const F2 n = f2_shfl_up(v, o);
        if (lane >= o) v = v + n;
    }
    return v;
}

__device__ __forceinline__ F2 warp_sum_f2(F2 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = v + F2{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---------------------------------------------------------------------------
// producer: warp kCW.  Lane 0 issues the copies; the whole warp resolves the
// next chunk, one step per fill, so that its loads overlap the copies of the
// current chunk.
// ---------------------------------------------------------------------------
struct Chunk {
    // 0: claim an index, 1: locate it, 2: load its metadata, 3: keep or
    // skip, 4: ready, 5: none left
    int stage;
    int c, q, r, g, b, k, Lb, d, rej;
    float u;  // bonus row: u'' of the bonus draw (position L_b)
};

__device__ void fetch_step(const VerifyArgs &a, const StreamShape &sh, Chunk &f, int epoch,
                           int lane) {
    if (f.stage == 0) {
        // the claim's round trip completes while the next fill is issued
        if (lane == 0) f.c = atomicAdd(&a.q_ctr[Q_CHUNK], 1);
        f.stage = 1;
    } else if (f.stage == 1) {
        f.c = __shfl_sync(0xffffffffu, f.c, 0);
        if (f.c >= sh.n_chunks) {
            f.stage = 5;
            return;
        }
        // packed row i of request b: index k = i - row_off[b] (k = L_b: the
        // bonus row)
        const int i = f.c / sh.cpr;
        f.g = f.c - i * sh.cpr;
        int off_b;
        f.b = find_request(a.row_off, a.B, i, lane, off_b);
        f.k = min(max(i - off_b, 0), a.gamma);
        f.r = min(i, sh.n_rows - 1);
        f.stage = 2;
    } else if (f.stage == 2) {
        // independent loads, one per lane; used a fill later
        int v = 0;
        if (lane == 0) v = a.L[f.b];
        else if (lane == 1 && f.k < a.gamma) v = a.draft_tokens[size_t(f.b) * a.gamma + f.k];
        f.d = v;  // parked in f.d per lane until the next step
        f.stage = 3;
    } else if (f.stage == 3) {
        const int v0 = __shfl_sync(0xffffffffu, f.d, 0);
        const int v1 = __shfl_sync(0xffffffffu, f.d, 1);
        f.Lb = min(max(v0, 0), a.gamma);
        f.q = f.k >= f.Lb;  // the bonus row
        f.d = f.q ? -1 : v1;
        f.u = 0.f;
        f.stage = 4;
    }
}

// A producer that gave up on a wait: let every copy it issued land before
// the CTA can leave (each is the only outstanding use of its stage).
__device__ void drain_copies(VSmem &sm, int fill, int lane) {
    if (lane == 0)
        for (int f = max(0, fill - kRing); f < fill; ++f)
            mbar_wait_bounded(&sm.full[f % kRing], (f / kRing) & 1, kDrainTimeoutNs);
    __syncwarp();
}

// ---------------------------------------------------------------------------
// consumer -> decider events
// ---------------------------------------------------------------------------
// Post an event (lane 0 of a consumer warp).  The caller has fenced its
// global writes; the FIFO store is ordered after them.
__device__ void post_event(const VerifyArgs &a, VSmem &sm, int ev) {
    const int pos = atomicAdd(&sm.fifo_tail, 1);
    if (pos - ld_vol(&sm.fifo_head) >= kFifo) {
        const uint64_t t0 = global_timer_ns();
        while (pos - ld_vol(&sm.fifo_head) >= kFifo) {
            if (global_timer_ns() - t0 > a.wait_ns) {
                atomicOr(a.status, kStatusQueueTimeout);
                return;
            }
            __nanosleep(64);
        }
    }
    __threadfence_block();
    st_vol(&sm.fifo[pos & (kFifo - 1)], ev);
}

// The producer's books.  A stage it takes back from the consumers is done,
// records included: the warp that writes a chunk's record releases the stage
// after writing it.  A decision chunk is then counted towards its request with
// a device atomic; the count comes back while the next fill is issued, and if
// it completed the request's decision rows the request goes to the CTA's
// decider (shared-memory FIFO).  Counting when the work completes, not when a
// decider gets to it, keeps a busy decider from becoming the last arriver of
// other requests.
struct Books {
    int ev;      // event to post once the count is back (0: none)
    int old;     // the counter's value before our increment
    int target;  // chunks of the request
};

__device__ __forceinline__ void check_books(const VerifyArgs &a, VSmem &sm, Books &bk) {
    if (bk.ev != 0 && bk.old == bk.target - 1) post_event(a, sm, bk.ev);
    bk.ev = 0;
}

__device__ __forceinline__ void book_stage(const VerifyArgs &a, VSmem &sm, const TaskInfo &t,
                                           Books &bk, const StreamShape &sh) {
    check_books(a, sm, bk);
    int *cnt;
    if (t.type == T_RESID) {
        // a residual tile of the request's rejected row pair
        cnt = &a.r1_cnt[t.b];
        bk.target = a.nc;
        bk.ev = ev_make(EV_R, 0, t.b);
    } else if (t.type == T_STREAM && t.flush) {
        if (t.k < t.Lb) {
            // a chunk of one of the request's decision rows
            cnt = &a.req_cnt[t.b];
            bk.target = t.Lb * sh.cpr;
            bk.ev = ev_make(EV_P, t.Lb, t.b);
        } else {
            // a chunk of its bonus row
            cnt = &a.bon_cnt[t.b];
            bk.target = sh.cprQ;
            bk.ev = ev_make(EV_Q, t.Lb, t.b);
        }
    } else {
        return;
    }
    __threadfence();
    bk.old = atomicAdd(cnt, 1);
}

// The end of a phase (the end marker is issued at `fill`): take back every
// stage still out, the marker's included, book what they held, and tell the
// decider that no more events will come.
__device__ bool finish_books(const VerifyArgs &a, VSmem &sm, int fill, int lane, Books &bk,
                             const StreamShape &sh) {
    for (int f = max(0, fill - kRing + 1); f <= fill; ++f) {
        int w = 1;
        if (lane == 0) w = mbar_wait_bounded(&sm.empty[f % kRing], (f / kRing) & 1, a.wait_ns);
        if (!__shfl_sync(0xffffffffu, w, 0)) {
            if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
            return false;
        }
        if (lane == 0) book_stage(a, sm, sm.task[f % kRing], bk, sh);
    }
    if (lane == 0) {
        check_books(a, sm, bk);
        // booked: the next phase's first fills take these stages back again
        for (int q = 0; q < kRing; ++q) sm.task[q].type = T_END;
        __threadfence_block();
        st_vol(&sm.prod_done, 1);
    }
    __syncwarp();
    return true;
}

// Take stage fill % kRing back from the consumers and fill it with task t
// (the whole producer warp; lane 0 issues).  A T_END task carries no copy:
// it ends the consumers' phase.  On a wait that gives up, lets the copies in
// flight land and returns false.
__device__ bool issue_fill(const VerifyArgs &a, VSmem &sm, uint8_t *ring, const TaskInfo &t,
                           int fill, int lane, Books &bk, const StreamShape &sh) {
    const int s = fill % kRing;
    if (fill >= kRing) {
        int w = 1;
        if (lane == 0) w = mbar_wait_bounded(&sm.empty[s], ((fill / kRing) - 1) & 1, a.wait_ns);
        if (!__shfl_sync(0xffffffffu, w, 0)) {
            if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
            drain_copies(sm, fill, lane);
            return false;
        }
        if (lane == 0) book_stage(a, sm, sm.task[s], bk, sh);
    }
    if (lane == 0) {
        sm.task[s] = t;
        uint64_t *bar = &sm.full[s];
        if (t.type == T_END) {
            mbar_arrive(bar);
        } else {
            uint8_t *dst = ring + s * kStageBytes;
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
        }
    }
    __syncwarp();
    return true;
}

// Phase 1: decision and bonus chunks.  Returns the index of the next fill.
__device__ int producer_stream(const VerifyArgs &a, VSmem &sm, uint8_t *ring,
                               const StreamShape &sh, int epoch, int lane, bool &ok) {
    Books bk{0, 0, 0};
    Chunk nx;
    nx.stage = 0;
    nx.c = 0;
    nx.d = 0;
    int cr = 0, cg = 0, cb = 0, ck = 0, cLb = 0, cd = -1, cj = 0, cj_end = 0, cq = 0;
    float cu = 0.f;
    bool in_chunk = false;
    for (int fill = 0;; ++fill) {
        TaskInfo t;
        t.type = T_END;
        if (!in_chunk && nx.stage != 5) {
            while (nx.stage < 4) fetch_step(a, sh, nx, epoch, lane);
            if (nx.stage == 4) {
                cq = nx.q;
                cr = nx.r;
                cg = nx.g;
                cb = nx.b;
                ck = nx.k;
                cLb = nx.Lb;
                cd = nx.d;
                cu = nx.u;
                const int C = cq ? sh.CTQ : sh.CT;
                cj = cg * C;
                cj_end = min(a.nc, cj + C);
                in_chunk = true;
                nx.stage = 0;
            }
        }
        if (in_chunk) {
            t.type = T_STREAM;
            t.r = cr;
            t.g = cg;
            t.b = cb;
            t.k = ck;
            t.Lb = cLb;
            t.d = cd;
            t.u_tok = cu;
            t.mode = 0;
            t.j = cj;
            t.pair = !a.greedy && !cq;
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
        }
        if (!issue_fill(a, sm, ring, t, fill, lane, bk, sh)) {
            ok = false;
            return fill;
        }
        if (t.type == T_END) {
            ok = finish_books(a, sm, fill, lane, bk, sh);
            return fill + 1;
        }
        // one step towards the next chunk
        if (nx.stage < 4) fetch_step(a, sh, nx, epoch, lane);
    }
}

// Phase 2: the tiles of every rejected row pair, tile t = blockIdx.x + i *
// gridDim.x of n_rej * nc.  Up to 32 tiles are located at once, one per lane
// (request, its draw state and row).  Returns the index of the next fill.
__device__ int producer_resid(const VerifyArgs &a, VSmem &sm, uint8_t *ring,
                              const StreamShape &sh, int fill, int lane, bool &ok) {
    Books bk{0, 0, 0};
    const int n_rej = min(max(ld_relaxed(&a.q_ctr[Q_NREJ]), 0), a.B);
    const int total = n_rej * a.nc;
    for (int base = blockIdx.x; base < total; base += 32 * int(gridDim.x)) {
        const int tl = base + lane * int(gridDim.x);
        TaskInfo mine;
        mine.type = T_END;
        if (tl < total) {
            const int rj = tl / a.nc;
            const int b = min(max(__ldcg(a.rej_list + rj), 0), a.B - 1);
            const DecideState st = load_state(a, b);
            const int r0 = __ldcg(a.row_off + b);
            mine.type = T_RESID;
            mine.b = b;
            mine.j = tl - rj * a.nc;
            mine.k = min(max(st.a, 0), a.gamma - 1);
            mine.r = min(max(r0 + mine.k, 0), sh.n_rows - 1);
            mine.Lb = 0;
            mine.g = 0;
            mine.d = -1;
            mine.flush = 0;
            mine.pair = 1;
            mine.y0 = mine.j * a.chunk_elems;
            mine.bytes = min(kChunkBytes, a.row_bytes - mine.j * kChunkBytes);
            mine.bytes2 = 0;
            mine.Mp = st.Mp;
            mine.Sp = st.Sp;
            mine.Mq = st.Mq;
            mine.Sq = st.Sq;
            mine.mode = st.mode;
            mine.u_tok = st.u_tok;
        }
        const int n = min(32, (total - base + int(gridDim.x) - 1) / int(gridDim.x));
        for (int l = 0; l < n; ++l, ++fill) {
            TaskInfo t;
            t.type = __shfl_sync(0xffffffffu, mine.type, l);
            t.b = __shfl_sync(0xffffffffu, mine.b, l);
            t.j = __shfl_sync(0xffffffffu, mine.j, l);
            t.k = __shfl_sync(0xffffffffu, mine.k, l);
            t.r = __shfl_sync(0xffffffffu, mine.r, l);
            t.Lb = 0;
            t.g = 0;
            t.d = -1;
            t.flush = 0;
            t.pair = 1;
            t.y0 = __shfl_sync(0xffffffffu, mine.y0, l);
            t.bytes = __shfl_sync(0xffffffffu, mine.bytes, l);
            t.bytes2 = 0;
            t.Mp = __shfl_sync(0xffffffffu, mine.Mp, l);
            t.Sp = __shfl_sync(0xffffffffu, mine.Sp, l);
            t.Mq = __shfl_sync(0xffffffffu, mine.Mq, l);
            t.Sq = __shfl_sync(0xffffffffu, mine.Sq, l);
            t.mode = __shfl_sync(0xffffffffu, mine.mode, l);
            t.u_tok = __shfl_sync(0xffffffffu, mine.u_tok, l);
            if (!issue_fill(a, sm, ring, t, fill, lane, bk, sh)) {
                ok = false;
                return fill;
            }
        }
    }
    TaskInfo t;
    t.type = T_END;
    if (!issue_fill(a, sm, ring, t, fill, lane, bk, sh)) {
        ok = false;
        return fill;
    }
    ok = finish_books(a, sm, fill, lane, bk, sh);
    return fill + 1;
}

// ---------------------------------------------------------------------------
// decisions and draws (warp-level)
// ---------------------------------------------------------------------------
// Draft tokens d_{b, lane} and d_{b, lane + 32} of a request, loaded once per
// decision (gamma <= 64).
struct Drafts {
    int t[2];
};

__device__ __forceinline__ Drafts load_drafts(const VerifyArgs &a, int b, int lane) {
    Drafts d;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int k = lane + 32 * i;
        d.t[i] = k < a.gamma ? __ldcg(a.draft_tokens + size_t(b) * a.gamma + k) : -1;
    }
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
        if (a.seq_lens_commit) a.seq_lens_commit[b] += acc + 1;
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// The two-level draw.  It runs once per request, latency-bound, on code that
// is cold in every SM when phase 3 starts, so it is kept compact: each block's
// mass is formed once by the lane that owns the block, one scan chooses the
// block, one the slot, and one vector's weights are formed a second time.
// ---------------------------------------------------------------------------
// What a slot record holds for a draw: the (max, sum) pair of p over the slot
// (a bonus row; the mass at the row's maximum M), the slot's residual mass,
// or its mass of p at the rejected row's own maximum.
enum : int { K_BONUS = 0, K_RESID = 1, K_P = 2 };

__device__ __forceinline__ float slot_mass(float2 x, int kind, float M, float scale) {
    if (kind == K_BONUS) return x.y > 0.f ? x.y * exp2_approx((x.x - M) * scale) : 0.f;
    return kind == K_RESID ? x.x : x.y;
}

// Mass of sampling block i: the two-float sum of its wpb slots.
__device__ __noinline__ F2 block_mass(const float2 *rec, int i, int wpb, int kind, float M,
                                      float scale) {
    float2 x[kCW];
#pragma unroll
    for (int w = 0; w < kCW; ++w)
        x[w] = w < wpb ? __ldcg(rec + size_t(i) * kCW + w) : make_float2(0.f, 0.f);
    F2 m = f2(0.f);
#pragma unroll
    for (int w = 0; w < kCW; ++w)
        if (w < wpb) m = m + f2(slot_mass(x[w], kind, M, scale));
    return m;
}

// The smallest index whose running mass exceeds `target` among the 32 lane
// values v (running sum `run` before them); -1 if none.  *last becomes the
// last index with positive mass seen so far, *run the running sum after them.
__device__ __forceinline__ int scan_pick(F2 v, bool live, F2 target, F2 &run, int base,
                                         int &last, int lane) {
    const F2 incl = run + warp_scan_incl(v, lane);
    const unsigned hit = __ballot_sync(0xffffffffu, live && f2_gt(incl, target));
    const unsigned pos = __ballot_sync(0xffffffffu, live && v.hi > 0.f);
    if (pos) last = base + 31 - __clz(pos);
    run = f2_shfl(incl, 31);
    return hit ? base + __ffs(hit) - 1 : -1;
}

// Draw weights of one 16-byte vector: p's unnormalised 2^((z - Mp) s) (a draw
// from p), or the normalised residual max(0, p - q).
template <typename T>
__device__ __forceinline__ void vec_weights(const uint4 &xv, const uint4 &yv, bool resid, float Mp,
                                            float iSp, float Mq, float iSq, float scale,
                                            float (&w)[Vec<T>::kElems]) {
    constexpr int VE = Vec<T>::kElems;
    float x[VE];
    Vec<T>::unpack(xv, x);
    if (resid) {
        float y[VE];
        Vec<T>::unpack(yv, y);
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

// The token of a draw inside one slot -- the ids [y0, y0 + 32 * kRunVec * VE)
// that one consumer warp covers in a tile: the smallest id whose running
// weight, counted from the slot's start, exceeds `target`.  Each lane owns a
// contiguous run of kRunVec vectors (one batch of loads); per-vector weights
// are summed pairwise and kept; runs are combined in two-float sums; the lane
// holding the crossing finds its vector from the kept sums and forms only that
// vector's weights again.  If rounding leaves no crossing, the last id with
// positive weight.
// What the draw needs of the launch, passed by value (a few registers): an
// out-of-line function taking the whole argument block by reference would
// copy it to the stack.
struct DrawCtx {
    const char *tgt, *dft;  // target and draft logits
    int row_bytes, gamma, nblk, chunk_elems;
    float scale;
};

__device__ __forceinline__ DrawCtx draw_ctx(const VerifyArgs &a) {
    return DrawCtx{static_cast<const char *>(a.target_logits),
                   static_cast<const char *>(a.draft_logits), a.row_bytes, a.gamma, a.nblk,
                   a.chunk_elems, a.scale};
}

template <typename T>
__device__ int slot_pick(const DrawCtx &a, const uint4 *tv, const uint4 *dv, bool resid,
                         int y0, F2 target, float Mp, float iSp, float Mq, float iSq, int lane) {
    constexpr int VE = Vec<T>::kElems;
    constexpr int kRunVec = 4;  // 32 lanes x 4 vectors: one warp's slot of a tile
    const int v_end = a.row_bytes / 16;
    const int v0 = y0 / VE + lane * kRunVec;
    uint4 xv[kRunVec], yv[kRunVec];
#pragma unroll
    for (int q = 0; q < kRunVec; ++q) {
        const bool in = v0 + q < v_end;
        xv[q] = in ? __ldcg(tv + v0 + q) : make_uint4(0, 0, 0, 0);
        yv[q] = in && resid ? __ldcg(dv + v0 + q) : make_uint4(0, 0, 0, 0);
    }
    float vs[kRunVec];
    float ls = 0.f;
#pragma unroll
    for (int q = 0; q < kRunVec; ++q) {
        float w[VE];
        vec_weights<T>(xv[q], yv[q], resid, Mp, iSp, Mq, iSq, a.scale, w);
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
        uint4 xs = xv[0], ys = yv[0];
#pragma unroll
        for (int q = 1; q < kRunVec; ++q)
            if (q == qsel) {
                xs = xv[q];
                ys = yv[q];
            }
        float w[VE];
        vec_weights<T>(xs, ys, resid, Mp, iSp, Mq, iSq, a.scale, w);
        float re = run_at;
        int lastpos = -1;
#pragma unroll
        for (int e = 0; e < VE; ++e) {
            re += w[e];
            if (pick < 0 && w[e] > 0.f) {
                lastpos = (v0 + qsel) * VE + e;
                if (f2_gt(excl + f2(re), target)) pick = (v0 + qsel) * VE + e;
            }
        }
        if (pick < 0) pick = lastpos >= 0 ? lastpos : v0 * VE;
    }
    return __shfl_sync(0xffffffffu, pick, lsel);
}

// The two-level draw of request b from the slot records `rec` ([nblk][kCW]):
// the smallest block whose running mass exceeds u_blk times the total, then
// within it the smallest slot whose running mass exceeds u_tok times the
// block's, then the id inside the slot (slot_pick).  Weights are p at target
// row r (K_BONUS: its maximum is taken from the records; K_P: Mp), or the
// residual of row r against draft row (b, dk) (K_RESID; a zero residual mass
// falls back to p of the same row).  The rows were streamed moments earlier.
template <typename T>
__device__ __noinline__ int draw_token(const DrawCtx a, int b, int r, int dk, int kind,
                                       const float2 *rec, float Mp, float Sp, float Mq, float Sq,
                                       float u_blk, float u_tok, int lane) {
    const int tpw = a.chunk_elems / kCW;
    const int wpb = kSampleBlock / tpw;
    const float scale = a.scale;
    float M = Mp;
    if (kind == K_BONUS) {
        float mb = -INFINITY;
#pragma unroll 1
        for (int i = lane; i < a.nblk; i += 32) {
            float2 x[kCW];
#pragma unroll
            for (int w = 0; w < kCW; ++w)
                x[w] = w < wpb ? __ldcg(rec + size_t(i) * kCW + w) : make_float2(0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kCW; ++w)
                if (w < wpb && x[w].y > 0.f) mb = fmaxf(mb, x[w].x);
        }
        M = warp_max(mb);
    }
    // Block masses (two blocks per lane kept for nblk <= 64) and their total.
    F2 keep0 = f2(0.f), keep1 = f2(0.f), total = f2(0.f);
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        total = f2(0.f);
#pragma unroll 1
        for (int t0 = 0; t0 < a.nblk; t0 += 32) {
            const int i = t0 + lane;
            const F2 m = i < a.nblk ? block_mass(rec, i, wpb, kind, M, scale) : f2(0.f);
            if (t0 == 0) keep0 = m;
            else if (t0 == 32) keep1 = m;
            total = total + warp_sum_f2(m);
        }
        if (kind != K_RESID || total.hi > 0.f) break;
        kind = K_P;  // no residual mass: draw from p of the same row
    }
    // The block.
    F2 target = f2_scale(total, u_blk), run = f2(0.f);
    int blk = -1, last = 0;
#pragma unroll 1
    for (int t0 = 0; t0 < a.nblk && blk < 0; t0 += 32) {
        const int i = t0 + lane;
        const F2 m = t0 == 0 ? keep0 : t0 == 32 ? keep1
                   : (i < a.nblk ? block_mass(rec, i, wpb, kind, M, scale) : f2(0.f));
        blk = scan_pick(m, i < a.nblk, target, run, t0, last, lane);
    }
    if (blk < 0) blk = last;
    // The slot within it: lane w holds slot w's mass.
    const float sm = lane < wpb ? slot_mass(__ldcg(rec + size_t(blk) * kCW + lane), kind, M, scale)
                                : 0.f;
    F2 bm = warp_sum_f2(f2(sm));
    target = f2_scale(bm, u_tok);
    run = f2(0.f);
    int wl = 0;
    int w = scan_pick(f2(sm), lane < wpb, target, run, 0, wl, lane);
    if (w < 0) w = wl;
    const F2 before = f2_shfl(f2_shfl_up(warp_scan_incl(f2(sm), lane), 1), w);
    const F2 inside = w > 0 ? target - before : target;
    // The token.
    const bool resid = kind == K_RESID;
    const uint4 *tv = reinterpret_cast<const uint4 *>(a.tgt + size_t(r) * a.row_bytes);
    const uint4 *dv = reinterpret_cast<const uint4 *>(
        resid ? a.dft + (size_t(b) * a.gamma + dk) * a.row_bytes : a.tgt);
    return slot_pick<T>(a, tv, dv, resid, blk * kSampleBlock + w * tpw, inside, M,
                        resid ? 1.f / Sp : 1.f, Mq, resid ? 1.f / Sq : 1.f, lane);
}

// The bonus draw of request b, every draft accepted: from p of row L_b
// (sampling; block and slot masses from the row's per-warp slots), or the
// argmax of row L_b (greedy; from its chunk records).
template <typename T>
__device__ void bonus_draw(const VerifyArgs &a, const StreamShape &sh, int b, int lane) {
    const int Lb = verify_len(a, b), r = a.row_off[b] + Lb;
    const Drafts dr = load_drafts(a, b, lane);
    int token;
    if (a.greedy) {
        float v = -INFINITY;
        int id = INT_MAX;
        const float4 *rec = a.rowrec + size_t(r) * a.grp_stride;
        for (int g = lane; g < sh.cprQ; g += 32) {
            const float4 x = __ldcg(rec + g);
            am_combine(v, id, x.x, __float_as_int(x.y));
        }
        warp_am_reduce(v, id);
        token = id;
    } else {
        const float3 un = uniforms_of(a.seed, b, Lb);
        token = draw_token<T>(draw_ctx(a), b, r, 0, K_BONUS, a.blkrec + size_t(b) * a.nblk * kCW,
                              0.f, 1.f, 0.f, 1.f, un.y, un.z, lane);
    }
    finish_request(a, b, Lb, token, dr, lane);
}

// Request b's decision rows (k < L_b) are all in: accept tests and outputs
// of the draft rows.  A rejection lists the request for the residual pass
// (sampling) or emits the row's argmax (greedy); with every draft accepted
// the bonus draw is due once the bonus row is in too: returns true when this
// call completes that join.  Loads that do not depend on one another are issued together: a
// decision runs while the streaming keeps L2 busy, and each dependent round
// trip costs microseconds.
template <typename T>
__device__ bool decide_request(const VerifyArgs &a, const StreamShape &sh, int b, int wpb,
                               int epoch, int lane) {
    // Round 1: lengths, offsets and draft tokens.  The request's count is
    // complete: reset it for the next launch.
    if (lane == 0) a.req_cnt[b] = 0;
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
        const int nrec = sh.cpr;
        const float4 *rec = a.rowrec + size_t(live ? r : r0) * a.grp_stride;
        constexpr int kRecBatch = 8;  // records per round of loads
        float4 x[kRecBatch];
#pragma unroll
        for (int u = 0; u < kRecBatch; ++u)
            x[u] = live && u < nrec ? __ldcg(rec + u) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float2 z = !a.greedy && live ? __ldcg(a.gath + r) : make_float2(0.f, 0.f);
        float u = 1.f, u1 = 0.f, u2 = 0.f;
        if (!a.greedy && live) {
            const float3 un = uniforms_of(a.seed, b, k);
            u = un.x;
            u1 = un.y;
            u2 = un.z;
        }
        float4 rr = a.greedy ? make_float4(-INFINITY, __int_as_float(INT_MAX), 0.f, 0.f)
                             : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        if (live) {
            for (int i0 = 0; i0 < nrec; i0 += kRecBatch) {
                if (i0 > 0) {
#pragma unroll
                    for (int v = 0; v < kRecBatch; ++v)
                        if (i0 + v < nrec) x[v] = __ldcg(rec + i0 + v);
                }
#pragma unroll
                for (int v = 0; v < kRecBatch; ++v) {
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
        if (a.greedy) {
            if (lane == 0) a.act[b] = A_NONE;
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
            a.act[b] = A_RESID;
            a.rej_list[atomicAdd(&a.q_ctr[Q_NREJ], 1)] = b;
        }
        return false;
    }
    // Every draft accepted: the bonus draw is due once the bonus row is in
    // too (join counter: whichever comes second queues it).
    int go = 0;
    if (lane == 0) {
        a.act[b] = A_BONUS;
        __threadfence();
        go = atomicAdd(&a.join[b], 1) == 1;
    }
    return __shfl_sync(0xffffffffu, go, 0);
}

// The residual draw of a rejected request (or, for a cap-accept window cut
// inside the accepted run, the draw from p at the window's row), from the
// per-slot masses of the residual pass.
template <typename T>
__device__ void finish_residual(const VerifyArgs &a, int b, int lane) {
    const DecideState st = load_state(a, b);
    const int r0 = a.row_off[b];
    const Drafts dr = load_drafts(a, b, lane);
    const int k = min(max(st.a, 0), a.gamma - 1);
    if (lane == 0) a.r1_cnt[b] = 0;  // the count is complete: reset it for the next launch
    const int token = draw_token<T>(draw_ctx(a), b, r0 + k, k, st.mode == D_RESID ? K_RESID : K_P,
                                    a.zrec + size_t(b) * a.nblk * kCW, st.Mp, st.Sp, st.Mq, st.Sq,
                                    st.u_blk, st.u_tok, lane);
    finish_request(a, b, st.a, token, dr, lane);
}

// ---------------------------------------------------------------------------
// consumers: warps 0 .. kCW-1
// ---------------------------------------------------------------------------
// Consumer warp of either streaming phase, from fill `fill`: returns the
// index of the fill after the phase's end.
template <typename T>
__device__ int consumer(const VerifyArgs &a, VSmem &sm, const uint8_t *ring,
                        const StreamShape &sh, int warp, int lane, int fill, int *fail) {
    constexpr int VE = Vec<T>::kElems;
    const float scale = a.scale;
    const int tpw = a.chunk_elems / kCW;  // tokens per warp in a tile
    const int vpw = tpw / VE;             // vectors per warp in a tile
    // Row accumulators of pair rows (sampling) / of every row (greedy),
    // carried across the tiles of a chunk.
    float mp = -INFINITY, sp = 0.f, mq = -INFINITY, sq = 0.f;
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (;; ++fill) {
        const int s = fill % kRing, n = fill / kRing, par = n & 1;
        if (!mbar_wait_backoff(&sm.full[s], n & 1, a.wait_ns)) {
            if (lane == 0) {
                atomicOr(a.status, kStatusWaitTimeout);
                atomicOr(fail, 1);
            }
            return fill;
        }
        const TaskInfo t = sm.task[s];
        if (t.type == T_END) {
            // the end of the phase: the stage goes back like any other
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
            return fill + 1;
        }
        const uint4 *tv = reinterpret_cast<const uint4 *>(ring + s * kStageBytes);
        const uint4 *dv = tv + kChunkBytes / 16;
        const int nvec = t.bytes / 16;
        const int v0 = min(nvec, warp * vpw), v1 = min(nvec, v0 + vpw);
        bool wrote = false;  // this warp wrote device memory another CTA will read

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
                for (int v = v0 + lane; v < v1; v += 32) {
                    float z[VE];
                    Vec<T>::unpack(tv[v], z);
                    online_update<VE>(mp, sp, z, scale);
                    Vec<T>::unpack(dv[v], z);
                    online_update<VE>(mq, sq, z, scale);
                }
                if (lane == 0) {
                    const int lo = t.y0 + v0 * VE, hi = t.y0 + v1 * VE;
                    if (t.d >= lo && t.d < hi) {
                        a.gath[t.r] = make_float2(Vec<T>::load1(tv, t.d - t.y0),
                                                  Vec<T>::load1(dv, t.d - t.y0));
                        wrote = true;
                    }
                }
            } else {
                // Bonus row: one (max, sum) slot per tile and warp -- the block
                // and slot masses of its draw.
                for (int h = 0; h < (t.bytes2 > 0 ? 2 : 1); ++h) {
                    const uint4 *xv = h ? dv : tv;
                    const int nv = (h ? t.bytes2 : t.bytes) / 16;
                    const int va = min(nv, warp * vpw), vb = min(nv, va + vpw);
                    float bm = -INFINITY, bs = 0.f;
                    for (int v = va + lane; v < vb; v += 32) {
                        float z[VE];
                        Vec<T>::unpack(xv[v], z);
                        online_update<VE>(bm, bs, z, scale);
                    }
                    warp_ms_reduce(bm, bs, scale);
                    const int y = t.y0 + h * a.chunk_elems + warp * tpw;
                    const int blk = y / kSampleBlock;
                    if (lane == 0 && blk < a.nblk) {
                        a.blkrec[(size_t(t.b) * a.nblk + blk) * kCW + (y % kSampleBlock) / tpw] =
                            make_float2(bm, bs);
                        wrote = true;
                    }
                }
            }
            // The stage has been read: hand it back before the bookkeeping,
            // except for the warp that writes a chunk's record (below).
            __syncwarp();
            if (!t.flush || !(a.greedy || t.pair)) {
                if (lane == 0) {
                    if (wrote) __threadfence();
                    mbar_arrive(&sm.empty[s]);
                }
                continue;
            }
            // End of a chunk: the eight warp partials become one record of
            // the row; the last warp writes it and only then releases the
            // stage, so the producer books the chunk once the record is in.
            {
                // The eight warp partials become one record of the row.
                float4 x;
                if (a.greedy) {
                    warp_am_reduce(bv, bi);
                    x = make_float4(bv, __int_as_float(bi), 0.f, 0.f);
                } else {
                    warp_ms_reduce(mp, sp, scale);
                    warp_ms_reduce(mq, sq, scale);
                    x = make_float4(mp, sp, mq, sq);
                }
                mp = mq = bv = -INFINITY;
                sp = sq = 0.f;
                bi = INT_MAX;
                int last = 0;
                if (lane == 0) {
                    sm.part[s][par][warp] = x;
                    if (wrote) __threadfence();
                    else __threadfence_block();
                    last = atomicAdd(&sm.done[s][par], 1) == kCW - 1;
                    if (!last) mbar_arrive(&sm.empty[s]);
                }
                if (__shfl_sync(0xffffffffu, last, 0)) {
                    __threadfence_block();
                    float4 y = lane < kCW ? sm.part[s][par][lane]
                                          : (a.greedy ? make_float4(-INFINITY, __int_as_float(INT_MAX), 0.f, 0.f)
                                                      : make_float4(-INFINITY, 0.f, -INFINITY, 0.f));
                    if (a.greedy) {
                        int yi = __float_as_int(y.y);
                        warp_am_reduce(y.x, yi);
                        y.y = __int_as_float(yi);
                    } else {
                        warp_ms_reduce(y.x, y.y, scale);
                        warp_ms_reduce(y.z, y.w, scale);
                    }
                    if (lane == 0) {
                        sm.done[s][par] = 0;
                        a.rowrec[size_t(t.r) * a.grp_stride + t.g] = y;
                        mbar_arrive(&sm.empty[s]);  // release after the record
                    }
                }
            }
            __syncwarp();
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
            const int y = t.y0 + warp * tpw;
            const int blk = y / kSampleBlock;
            if (lane == 0) {
                if (blk < a.nblk)
                    a.zrec[(size_t(t.b) * a.nblk + blk) * kCW + (y % kSampleBlock) / tpw] =
                        make_float2(dr.hi + dr.lo, dp.hi + dp.lo);
                __threadfence();
                mbar_arrive(&sm.empty[s]);  // after the record: the producer books the tile
            }
            __syncwarp();
        }
    }
}

// ---------------------------------------------------------------------------
// draws queued in the CTA, and the warps that make them
// ---------------------------------------------------------------------------
// Queue a draw (the decider's lane 0; the decider is the only writer of the
// tail).  Returns false when the queue is full: the caller draws itself.
__device__ __forceinline__ bool push_job(VSmem &sm, int ev) {
    const int t = sm.job_tail;
    if (t - ld_vol(&sm.job_head) >= kJobs) return false;
    st_vol(&sm.jobs[t & (kJobs - 1)], ev);
    __threadfence_block();
    st_vol(&sm.job_tail, t + 1);
    return true;
}

// Take a queued draw (lane 0 of any warp): its event code, or 0.
__device__ __forceinline__ int claim_job(VSmem &sm) {
    const int h = ld_vol(&sm.job_head);
    if (h >= ld_vol(&sm.job_tail)) return 0;
    if (atomicCAS(&sm.job_head, h, h + 1) != h) return 0;  // another warp took it
    __threadfence_block();
    return ld_vol(&sm.jobs[h & (kJobs - 1)]);
}

template <typename T>
__device__ __forceinline__ void run_job(const VerifyArgs &a, const StreamShape &sh, int ev,
                                        int lane) {
    __threadfence();
    if (((ev >> 24) & 3) == EV_R) finish_residual<T>(a, ev & 0xffff, lane);
    else bonus_draw<T>(a, sh, ev & 0xffff, lane);
}

// A warp done with its part of the phase makes queued draws until the
// decider has queued the last one.
template <typename T>
__device__ void helper(const VerifyArgs &a, VSmem &sm, const StreamShape &sh, int lane,
                       int *fail) {
    uint64_t t0 = global_timer_ns();
    unsigned ns = 64;
    for (;;) {
        int ev = 0, quit = 0;
        if (lane == 0) {
            ev = claim_job(sm);
            if (ev == 0) {
                if (ld_vol(&sm.no_more) && ld_vol(&sm.job_head) >= ld_vol(&sm.job_tail)) {
                    quit = 1;
                } else if (global_timer_ns() - t0 > a.wait_ns) {
                    atomicOr(a.status, kStatusQueueTimeout);
                    atomicOr(fail, 1);
                    quit = 1;
                }
            }
        }
        ev = __shfl_sync(0xffffffffu, ev, 0);
        if (ev != 0) {
            run_job<T>(a, sh, ev, lane);
            if (lane == 0) {
                t0 = global_timer_ns();
                ns = 64;
            }
            continue;
        }
        if (__shfl_sync(0xffffffffu, quit, 0)) return;
        if (lane == 0) {
            __nanosleep(ns);
            ns = min(ns * 2, 512u);
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// decider: warp kCW + 1
// ---------------------------------------------------------------------------
// Works through the events its producer posts, in order: decide a request
// whose decision rows are in; queue the bonus draw of a request whose bonus
// row is in and whose drafts were all accepted (join counter); queue the
// residual draw of a request whose residual tiles are in.  Between events it
// makes queued draws itself.  Returns once the producer has booked every unit
// of the phase, the FIFO is empty and every draw is queued or made.
template <typename T>
__device__ void decider(const VerifyArgs &a, VSmem &sm, const StreamShape &sh, int epoch,
                        int lane, int *fail) {
    const int wpb = kSampleBlock / (a.chunk_elems / kCW);
    uint64_t t_last = global_timer_ns();
    unsigned ns = 32;
    for (;;) {
        int v = 0, h = 0, job = 0, done = 0;
        if (lane == 0) {
            h = ld_vol(&sm.fifo_head);
            v = ld_vol(&sm.fifo[h & (kFifo - 1)]);
            if (v != 0) {
                st_vol(&sm.fifo[h & (kFifo - 1)], 0);
                __threadfence_block();
                st_vol(&sm.fifo_head, h + 1);
            } else if ((job = claim_job(sm)) != 0) {
                // a queued draw while no event waits
            } else if (ld_vol(&sm.prod_done) && ld_vol(&sm.fifo_tail) == h) {
                done = 1;  // every unit booked, every event handled, every draw taken
                st_vol(&sm.no_more, 1);
            } else if (global_timer_ns() - t_last > a.wait_ns) {
                atomicOr(a.status, kStatusQueueTimeout);
                atomicOr(fail, 1);
                st_vol(&sm.no_more, 1);
                done = 1;
            }
        }
        v = __shfl_sync(0xffffffffu, v, 0);
        job = __shfl_sync(0xffffffffu, job, 0);
        if (__shfl_sync(0xffffffffu, done, 0)) return;
        if (v != 0) {
            const int type = (v >> 24) & 3, Lb = (v >> 16) & 127, b = v & 0xffff;
            __threadfence();
            int draw = 0;  // a draw now due: queue it
            if (type == EV_P) {
                draw = decide_request<T>(a, sh, b, wpb, epoch, lane) ? ev_make(EV_Q, Lb, b) : 0;
            } else if (type == EV_Q) {
                if (lane == 0 && (Lb == 0 || atomicAdd(&a.join[b], 1) == 1)) draw = v;
                draw = __shfl_sync(0xffffffffu, draw, 0);
            } else {
                draw = v;
            }
            if (draw != 0) {
                int queued = 0;
                if (lane == 0) queued = push_job(sm, draw);
                if (!__shfl_sync(0xffffffffu, queued, 0)) run_job<T>(a, sh, draw, lane);
            }
            if (lane == 0) {
                t_last = global_timer_ns();
                ns = 32;
            }
            continue;
        }
        if (job != 0) {
            run_job<T>(a, sh, job, lane);
            if (lane == 0) {
                t_last = global_timer_ns();
                ns = 32;
            }
            continue;
        }
        if (lane == 0) {
            __nanosleep(ns);
            ns = min(ns * 2, 256u);
        }
        __syncwarp();
    }
}

// Grid-wide barrier of the cooperative launch (every CTA is resident).  The
// generation is read before arriving, so the last arrival's increment cannot
// be missed.  Gives up after wait_ns (status bit) and returns false.
__device__ bool grid_sync(const VerifyArgs &a, int *s_ok) {
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const int gen = ld_relaxed(&a.q_ctr[Q_BARGEN]);
        __threadfence();
        if (atomicAdd(&a.q_ctr[Q_BAR], 1) == int(gridDim.x) - 1) {
            a.q_ctr[Q_BAR] = 0;
            __threadfence();
            atomicAdd(&a.q_ctr[Q_BARGEN], 1);
        } else {
            const uint64_t t0 = global_timer_ns();
            unsigned ns = 32;
            while (ld_acquire(&a.q_ctr[Q_BARGEN]) == gen) {
                if (global_timer_ns() - t0 > a.wait_ns) {
                    atomicOr(a.status, kStatusQueueTimeout);
                    ok = 0;
                    break;
                }
                __nanosleep(ns);
                ns = min(ns * 2, 128u);
            }
        }
        __threadfence();
        *s_ok = ok;
    }
    __syncthreads();
    return *s_ok != 0;
}

template <typename T>
__global__ void __launch_bounds__(kVerifyThreads, 2) verify_kernel(const VerifyArgs a) {
    extern __shared__ __align__(1024) uint8_t ring[];
    __shared__ VSmem sm;
    __shared__ int s_fail, s_bar, s_last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int epoch = ld_relaxed(&a.q_ctr[Q_EPOCH]) + 1;
    if (tid < kRing) {
        mbar_init(&sm.full[tid], 1);
        mbar_init(&sm.empty[tid], kCW);
        sm.done[tid][0] = 0;
        sm.done[tid][1] = 0;
    }
    if (tid < kFifo) sm.fifo[tid] = 0;
    if (tid == 0) {
        sm.fifo_tail = 0;
        sm.fifo_head = 0;
        sm.job_tail = 0;
        sm.job_head = 0;
        sm.no_more = 0;
        sm.prod_done = 0;
        s_fail = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const StreamShape sh = stream_shape(a);
    int fill = 0;  // the ring's next fill (producer and consumers keep it in step)

    // Phase 1: stream the decision and bonus rows; decide each request and
    // draw the bonus tokens.
    if (warp == kCW) {
        bool ok = true;
        fill = producer_stream(a, sm, ring, sh, epoch, lane, ok);
        if (!ok && lane == 0) atomicOr(&s_fail, 1);
        helper<T>(a, sm, sh, lane, &s_fail);
    } else if (warp == kCW + 1) {
        decider<T>(a, sm, sh, epoch, lane, &s_fail);
    } else {
        fill = consumer<T>(a, sm, ring, sh, warp, lane, 0, &s_fail);
        helper<T>(a, sm, sh, lane, &s_fail);
    }
    __syncthreads();
    if (tid == 0) {
        sm.prod_done = 0;
        sm.no_more = 0;
    }
    // Phase 2, once every request is decided: the residual tiles of the
    // rejected row pairs, each with its blocks' in-block picks; the CTA that
    // completes a request's tiles draws its token.  A CTA whose ring gave up
    // starts no copy.
    if (!grid_sync(a, &s_bar)) atomicOr(&s_fail, 1);
    if (ld_relaxed(&a.q_ctr[Q_NREJ]) > 0) {
        if (warp == kCW + 1) {
            decider<T>(a, sm, sh, epoch, lane, &s_fail);
        } else {
            if (!s_fail) {
                if (warp == kCW) {
                    bool ok = true;
                    fill = producer_resid(a, sm, ring, sh, fill, lane, ok);
                    if (!ok && lane == 0) atomicOr(&s_fail, 1);
                } else {
                    fill = consumer<T>(a, sm, ring, sh, warp, lane, fill, &s_fail);
                }
            } else if (warp == kCW && lane == 0) {
                st_vol(&sm.prod_done, 1);  // nothing streams here: let the decider go
            }
            helper<T>(a, sm, sh, lane, &s_fail);
        }
    }

    __syncthreads();
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(&a.q_ctr[Q_EXITED], 1) == int(gridDim.x) - 1;
    }
    __syncthreads();
    if (s_last) {
        // Every CTA is done.  Bonus-row counts of requests that rejected can
        // be partial, and joins of requests without drafts are never used:
        // these reset here.
        __threadfence();
        for (int b = tid; b < a.B; b += kVerifyThreads) {
            a.bon_cnt[b] = 0;
            a.join[b] = 0;
        }
    }
    if (s_last && tid == 0) {
        // Reset the counters for the next launch.
        __threadfence();
        a.q_ctr[Q_CHUNK] = 0;
        a.q_ctr[Q_NREJ] = 0;
        a.q_ctr[Q_EXITED] = 0;
        a.q_ctr[Q_EPOCH] = epoch;
        if (a.audit_totals) {
            a.audit_totals[0] = atomicExch(&a.q_ctr[Q_AFULL], 0);
            a.audit_totals[1] = atomicExch(&a.q_ctr[Q_ACOMMIT], 0);
        }
        __threadfence();
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
    // Cooperative launch: the phases are separated by grid barriers, so every
    // CTA of the grid must be resident at once.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kVerifyThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (logit_bf16) return cudaLaunchKernelEx(&cfg, verify_kernel<uint16_t>, a);
    return cudaLaunchKernelEx(&cfg, verify_kernel<float>, a);
}

}  // namespace dspark
