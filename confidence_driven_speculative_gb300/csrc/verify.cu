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
// and every kept draft row (sum L) is read once, V logits each.
//
//  * One persistent cooperative grid, 2 CTAs per SM.  Each CTA is one
//    producer warp and 8 consumer warps.  The producer's lane 0 fills a
//    3-stage shared-memory ring with 1-D bulk TMA copies (cp.async.bulk),
//    each stage completing on a "full" mbarrier with a byte count; consumers
//    release a stage on an "empty" mbarrier (one arrival per warp).  There is
//    no block-wide barrier in the loop: warps only meet through mbarriers and
//    a per-stage shared counter that elects the last warp of each stage.
//  * Stream tasks: (packed row r, 16 KB vocab tile j).  Row r of request b
//    at index k < L_b is a pair (target row r, draft row (b, k)); k = L_b is
//    the bonus row.  Each CTA takes a contiguous range of stream tasks.  Each
//    consumer warp folds its eighth of the tile into an online (max, sum) of
//    2^(z * log2(e)/Tm) for p and q (greedy: max and lowest argmax); the
//    stage's last warp merges the eight partials into one record per
//    4096-token sampling block and counts the tile for its request.
//  * The warp that counts a request's last tile decides it: accept tests
//    (Philox uniforms), p(d)/q(d) outputs, and the draw of the emitted token
//    in two levels, a 4096-id block by mass (u') then an id inside it (u'').
//    A bonus draw takes block masses from the records and pushes one "pick"
//    job; a residual draw pushes one "residual mass" job per tile of the
//    rejecting row pair (read again while it is still in L2), and the last
//    of those pushes the pick.  Jobs go to a device-wide queue that every
//    producer serves before its own stream tasks, so this work is spread over
//    the whole GPU and flows through the same TMA ring.
//  * Every wait is bounded (mbarrier waits and queue polls give up after 2 s
//    and set a status bit); counters reset themselves at the end of the
//    launch, so the kernel can be replayed.
#include <climits>

#include "dspark_internal.cuh"

namespace dspark {
namespace {

constexpr int kCW = kConsumerWarps;
constexpr int kStageBytes = 2 * kChunkBytes;  // target tile + draft tile
constexpr size_t kSmemBytes = size_t(kStages) * kStageBytes;

enum : int { T_EXIT = 0, T_STREAM = 1, T_RESID = 2, T_PICK = 3, T_DECIDE = 4, T_RBLOCK = 5 };
enum : int { D_BONUS = 0, D_RESID = 1, D_FALLBACK = 2 };
enum : int { Q_HEAD = 0, Q_TAIL = 1, Q_FINISHED = 2, Q_EXITED = 3, Q_EPOCH = 4 };

struct TaskInfo {
    int type;   // T_*
    int b;      // request
    int r;      // packed target row read by the stage
    int k;      // draft index of the draft row (pair) / of the drawn row
    int Lb;     // verify length of request b
    int j;      // stream / residual: tile index; pick: sampling block index
    int y0;     // first token id of the stage
    int bytes;  // bytes per row in the stage
    int pair;   // a draft row sits in the second half of the stage
    int d;      // drafted id of a stream pair (its gather target)
};

struct VSmem {
    uint64_t full[kStages], empty[kStages];
    TaskInfo task[kStages];
    float4 wpart[kStages][kCW];
    double wd[kStages][kCW];
    float2 gath[kStages];
    int gflag[kStages];
    int done[kStages];
};

// ---------------------------------------------------------------------------
// small memory-model helpers
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
__device__ __forceinline__ void st_release(int *p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
                 : "memory");
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

// Fold one vector of logits into a running (max, sum of 2^((z - max) * s)).
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
#pragma unroll
    for (int e = 0; e < VE; ++e) s += exp2_approx(fmaf(x[e], scale, -ms));
}

// Inclusive warp scan in double (lane order).
__device__ __forceinline__ double warp_scan_incl(double v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// ---------------------------------------------------------------------------
// job queue
// ---------------------------------------------------------------------------
__device__ void push_jobs(const VerifyArgs &a, int type, int b, int first, int count,
                          int epoch) {
    const int pos = atomicAdd(&a.q_ctr[Q_TAIL], count);
    for (int i = 0; i < count; ++i)
        if (pos + i < a.qcap) a.q_job[pos + i] = make_int2((type << 24) | b, first + i);
    __threadfence();
    for (int i = 0; i < count; ++i)
        if (pos + i < a.qcap) st_release(&a.q_ready[pos + i], epoch);
}

// Turn a queued job into the stage it reads (decide jobs read nothing).
__device__ TaskInfo decode_job(const VerifyArgs &a, int2 jb) {
    TaskInfo t;
    t.type = jb.x >> 24;
    t.b = jb.x & 0xffffff;
    t.j = jb.y;
    t.d = -1;
    t.Lb = verify_len(a, t.b);
    t.r = t.k = t.y0 = t.bytes = t.pair = 0;
    if (t.type == T_DECIDE || t.type == T_RBLOCK) return t;
    const DecideState st = load_state(a, t.b);
    const int r0 = a.row_off[t.b];
    if (t.type == T_RESID) {
        t.k = st.a;
        t.r = r0 + st.a;
        t.pair = 1;
        t.y0 = t.j * a.chunk_elems;
        t.bytes = min(kChunkBytes, a.row_bytes - t.j * kChunkBytes);
    } else {
        t.k = st.mode == D_BONUS ? t.Lb : st.a;
        t.r = r0 + t.k;
        t.pair = st.mode == D_RESID;
        t.y0 = t.j * kSampleBlock;
        t.bytes = min(kSampleBlock * a.elem_bytes, a.row_bytes - t.y0 * a.elem_bytes);
    }
    return t;
}

// Per-row metadata of the packed rows, fetched ahead of use.
struct RowMeta {
    int b, k, Lb, d;
};

__device__ __forceinline__ void row_ids(const VerifyArgs &a, int r, int n_rows, int &b, int &k) {
    b = r < n_rows ? a.row_req[r] : 0;
    k = r < n_rows ? a.row_k[r] : 0;
}

__device__ __forceinline__ RowMeta row_meta(const VerifyArgs &a, int b, int k) {
    RowMeta m;
    m.b = b;
    m.k = k;
    m.Lb = verify_len(a, b);
    m.d = k < a.gamma ? a.draft_tokens[size_t(b) * a.gamma + k] : -1;
    return m;
}

__device__ __forceinline__ TaskInfo stream_task(const VerifyArgs &a, const RowMeta &m, int r,
                                                int j) {
    TaskInfo t;
    t.type = T_STREAM;
    t.r = r;
    t.j = j;
    t.b = m.b;
    t.k = m.k;
    t.Lb = m.Lb;
    t.d = m.d;
    t.pair = !a.greedy && m.k < m.Lb;
    t.y0 = j * a.chunk_elems;
    t.bytes = min(kChunkBytes, a.row_bytes - j * kChunkBytes);
    return t;
}

// ---------------------------------------------------------------------------
// producer: lane 0 of the last warp.  Besides feeding the ring it keeps the
// books of the stages it gets back: stream tiles are counted per request
// locally and added to the request's counter once per request change (one
// fence and one atomic instead of one per tile); a request whose count
// completes is pushed as a decide job, so no consumer ever stalls on a
// device-wide fence or atomic while it holds a stage.
// ---------------------------------------------------------------------------
struct Books {
    int acc_b, acc_n, acc_total;
};

__device__ void flush_books(const VerifyArgs &a, Books &bk, int epoch) {
    if (bk.acc_n == 0) return;
    __threadfence();
    const int old = atomicAdd(&a.req_cnt[bk.acc_b], bk.acc_n);
    if (old + bk.acc_n == bk.acc_total) push_jobs(a, T_DECIDE, bk.acc_b, 0, 1, epoch);
    bk.acc_n = 0;
}

__device__ void account(const VerifyArgs &a, Books &bk, const TaskInfo &t, int epoch) {
    if (t.type == T_STREAM) {
        if (t.b != bk.acc_b) {
            flush_books(a, bk, epoch);
            bk.acc_b = t.b;
            bk.acc_total = (t.Lb + 1) * a.nc;
        }
        ++bk.acc_n;
    } else if (t.type == T_RESID) {
        __threadfence();
        if (atomicAdd(&a.r1_cnt[t.b], 1) == a.nc - 1) push_jobs(a, T_RBLOCK, t.b, 0, 1, epoch);
    }
}

// Wait for every fill below `upto` to come back from the consumers and book it.
__device__ bool reclaim(const VerifyArgs &a, VSmem &sm, Books &bk, int &booked, int upto,
                        int epoch) {
    for (; booked < upto; ++booked) {
        const int s = booked % kStages;
        if (!mbar_wait_bounded(&sm.empty[s], (booked / kStages) & 1)) {
            atomicOr(a.status, kStatusWaitTimeout);
            return false;
        }
        account(a, bk, sm.task[s], epoch);
    }
    return true;
}

__device__ void producer(const VerifyArgs &a, VSmem &sm, uint8_t *ring, long long s_lo,
                         long long s_hi, int n_rows, int epoch) {
    constexpr int kQueuePoll = 4;  // look at the queue every few stream tiles
    long long s_next = s_lo;
    // Row metadata pipeline: `cur` in use, `nxt` loaded, ids of the row after
    // that in flight, so no global load latency sits between two tiles.
    int r_cur = int(s_lo / a.nc), j_cur = int(s_lo - (long long)r_cur * a.nc);
    RowMeta cur{}, nxt{};
    int nb = 0, nk = 0;
    if (s_lo < s_hi) {
        int b, k;
        row_ids(a, r_cur, n_rows, b, k);
        cur = row_meta(a, b, k);
        row_ids(a, r_cur + 1, n_rows, b, k);
        nxt = row_meta(a, b, k);
        row_ids(a, r_cur + 2, n_rows, nb, nk);
    }
    Books bk{-1, 0, 0};
    int booked = 0;
    int pending = -1;  // a queue index this CTA has claimed but not yet seen filled
    int since_poll = kQueuePoll;
    for (int fill = 0;; ++fill) {
        TaskInfo t;
        t.type = T_EXIT;
        bool have = false, ok = true;
        if (since_poll >= kQueuePoll || s_next >= s_hi) {
            since_poll = 0;
            if (pending < 0 && ld_relaxed(&a.q_ctr[Q_HEAD]) < ld_relaxed(&a.q_ctr[Q_TAIL]))
                pending = atomicAdd(&a.q_ctr[Q_HEAD], 1);
            if (pending >= 0 && pending < a.qcap && ld_acquire(&a.q_ready[pending]) == epoch) {
                t = decode_job(a, __ldcg(a.q_job + pending));
                pending = -1;
                have = true;
            }
        }
        if (!have && s_next < s_hi) {
            t = stream_task(a, cur, r_cur, j_cur);
            have = true;
            ++s_next;
            ++since_poll;
            if (++j_cur == a.nc) {
                j_cur = 0;
                ++r_cur;
                cur = nxt;
                nxt = row_meta(a, nb, nk);
                row_ids(a, r_cur + 2, n_rows, nb, nk);
            }
        }
        if (!have) {
            // Own tiles are done: book everything in flight, then serve the
            // queue until every request has finished.
            ok = reclaim(a, sm, bk, booked, fill, epoch);
            flush_books(a, bk, epoch);
            if (pending < 0) pending = atomicAdd(&a.q_ctr[Q_HEAD], 1);
            const uint64_t t0 = global_timer_ns();
            unsigned ns = 64;
            while (ok) {
                if (pending < a.qcap && ld_acquire(&a.q_ready[pending]) == epoch) {
                    t = decode_job(a, __ldcg(a.q_job + pending));
                    pending = -1;
                    have = true;
                    break;
                }
                if (ld_acquire(&a.q_ctr[Q_FINISHED]) >= a.B) break;
                if (global_timer_ns() - t0 > kWaitTimeoutNs) {
                    atomicOr(a.status, kStatusQueueTimeout);
                    break;
                }
                __nanosleep(ns);
                ns = min(ns * 2, 2048u);
            }
        }
        const int s = fill % kStages;
        if (ok) ok = reclaim(a, sm, bk, booked, fill - kStages + 1, epoch);
        if (!have || !ok) t.type = T_EXIT;
        sm.task[s] = t;
        if (t.type == T_EXIT || t.bytes == 0) {
            mbar_arrive(&sm.full[s]);  // a stage without data
            if (t.type == T_EXIT) return;
            continue;
        }
        uint8_t *dst = ring + s * kStageBytes;
        uint64_t *bar = &sm.full[s];
        const char *tsrc = static_cast<const char *>(a.target_logits) +
                           size_t(t.r) * a.row_bytes + size_t(t.y0) * a.elem_bytes;
        mbar_arrive_expect_tx(bar, uint32_t(t.bytes) * (t.pair ? 2u : 1u));
        bulk_g2s(dst, tsrc, uint32_t(t.bytes), bar);
        if (t.pair) {
            const char *dsrc = static_cast<const char *>(a.draft_logits) +
                               (size_t(t.b) * a.gamma + t.k) * size_t(a.row_bytes) +
                               size_t(t.y0) * a.elem_bytes;
            bulk_g2s(dst + kChunkBytes, dsrc, uint32_t(t.bytes), bar);
        }
    }
}

// ---------------------------------------------------------------------------
// request completion (warp-level)
// ---------------------------------------------------------------------------
__device__ void finish_request(const VerifyArgs &a, int b, int acc, int token, int lane) {
    const int g1 = a.gamma + 1;
    for (int j = lane; j < g1; j += 32) {
        int v = -1;
        if (j < acc) v = a.draft_tokens[size_t(b) * a.gamma + j];
        else if (j == acc) v = token;
        a.out_tokens[size_t(b) * g1 + j] = v;
    }
    if (lane == 0) {
        a.accept_len[b] = acc;
        a.num_emitted[b] = acc + 1;
        if (a.seq_lens_commit) a.seq_lens_commit[b] += acc + 1;
        a.req_cnt[b] = 0;
        a.r1_cnt[b] = 0;
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) atomicAdd(&a.q_ctr[Q_FINISHED], 1);
}

// Choose a sampling block: the smallest i whose running mass exceeds
// u * total; the last block with positive mass if rounding leaves no
// crossing.  Warp-level; mass(i) is evaluated by the lane that owns i.
template <typename F>
__device__ int choose_block(int nblk, float u, F mass, int lane) {
    double total = 0.0;
    for (int t0 = 0; t0 < nblk; t0 += 32) {
        const int i = t0 + lane;
        const double incl = warp_scan_incl(i < nblk ? double(mass(i)) : 0.0, lane);
        total += __shfl_sync(0xffffffffu, incl, 31);
    }
    const double target = double(u) * total;
    double run = 0.0;
    int last_pos = 0;
    for (int t0 = 0; t0 < nblk; t0 += 32) {
        const int i = t0 + lane;
        const double v = i < nblk ? double(mass(i)) : 0.0;
        const double incl = run + warp_scan_incl(v, lane);
        const unsigned hit = __ballot_sync(0xffffffffu, i < nblk && incl > target);
        if (hit) return t0 + __ffs(hit) - 1;
        const unsigned pos = __ballot_sync(0xffffffffu, i < nblk && v > 0.0);
        if (pos) last_pos = t0 + 31 - __clz(pos);
        run = __shfl_sync(0xffffffffu, incl, 31);
    }
    return last_pos;
}

// Decide request b once all its stream tiles are in (warp-level).
__device__ void decide_request(const VerifyArgs &a, int b, int epoch, int lane) {
    const int Lb = verify_len(a, b), r0 = a.row_off[b], d0 = a.draft_off[b];
    const int nb = a.nblk;
    const float scale = a.scale;
    int ab = Lb;                                   // first rejected draft (L_b: none)
    float Mp = 0.f, Sp = 0.f, Mq = 0.f, Sq = 0.f;  // normalisers of row a_b (sampling)
    float Mbonus = 0.f;
    int g_tok = 0;
    // One lane per row k (two rounds when gamma >= 32); each lane folds the
    // row's block records, loads issued eight at a time.
    for (int base = 0; base <= Lb; base += 32) {
        const int k = base + lane;
        const bool live = k <= Lb;
        const float4 *rec = a.rec + size_t(r0 + (live ? k : 0)) * a.nblk_stride;
        bool accept = false;
        if (a.greedy) {
            float bv = -INFINITY;
            int bi = INT_MAX;
            if (live) {
                for (int i0 = 0; i0 < nb; i0 += 8) {
                    float4 x[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        x[u] = i0 + u < nb ? __ldcg(rec + i0 + u)
                                           : make_float4(-INFINITY, __int_as_float(INT_MAX), 0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < 8; ++u) am_combine(bv, bi, x[u].x, __float_as_int(x[u].y));
                }
                if (k < Lb) {
                    accept = a.draft_tokens[size_t(b) * a.gamma + k] == bi;
                    a.p_tok[d0 + k] = 0.f;
                    a.q_tok[d0 + k] = 0.f;
                }
            }
            const unsigned acc = __ballot_sync(0xffffffffu, live && k < Lb && accept);
            const unsigned rows = __ballot_sync(0xffffffffu, live && k < Lb);
            const unsigned rej = rows & ~acc;
            if (ab == Lb && rej) ab = base + __ffs(rej) - 1;
            const int src = ab - base;
            const int g = __shfl_sync(0xffffffffu, bi, src >= 0 && src < 32 ? src : 0);
            if (src >= 0 && src < 32) g_tok = g;
        } else {
            float mp = -INFINITY, sp = 0.f, mq = -INFINITY, sq = 0.f;
            if (live) {
                for (int i0 = 0; i0 < nb; i0 += 8) {
                    float4 x[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        x[u] = i0 + u < nb ? __ldcg(rec + i0 + u)
                                           : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        ms_combine(mp, sp, x[u].x, x[u].y, scale);
                        ms_combine(mq, sq, x[u].z, x[u].w, scale);
                    }
                }
                if (k < Lb) {
                    const int dt = a.draft_tokens[size_t(b) * a.gamma + k];
                    float p = 0.f, q = 0.f, ratio = 0.f;
                    if (dt >= 0 && dt < a.V) {
                        const float2 z = __ldcg(a.gath + r0 + k);
                        p = exp2_approx((z.x - mp) * scale) / sp;
                        q = exp2_approx((z.y - mq) * scale) / sq;
                        ratio = q > 0.f ? fminf(1.f, p / q) : 1.f;
                    }
                    float u, ub, ut;
                    step_uniforms(a.seed, b, k, u, ub, ut);
                    accept = u < ratio;
                    a.p_tok[d0 + k] = p;
                    a.q_tok[d0 + k] = q;
                }
            }
            const unsigned acc = __ballot_sync(0xffffffffu, live && k < Lb && accept);
            const unsigned rows = __ballot_sync(0xffffffffu, live && k < Lb);
            const unsigned rej = rows & ~acc;
            if (ab == Lb && rej) ab = base + __ffs(rej) - 1;
            const int src = ab - base;
            const int sl = src >= 0 && src < 32 ? src : 0;
            const float m1 = __shfl_sync(0xffffffffu, mp, sl), s1 = __shfl_sync(0xffffffffu, sp, sl);
            const float m2 = __shfl_sync(0xffffffffu, mq, sl), s2 = __shfl_sync(0xffffffffu, sq, sl);
            if (src >= 0 && src < 32) {
                Mp = m1;
                Sp = s1;
                Mq = m2;
                Sq = s2;
            }
            const int bsrc = Lb - base;
            const float mb = __shfl_sync(0xffffffffu, mp, bsrc >= 0 && bsrc < 32 ? bsrc : 0);
            if (bsrc >= 0 && bsrc < 32) Mbonus = mb;
        }
    }
    if (a.greedy) {
        finish_request(a, b, ab, g_tok, lane);
        return;
    }
    float u, ub, ut;
    step_uniforms(a.seed, b, ab, u, ub, ut);
    DecideState st;
    st.a = ab;
    st.u_blk = ub;
    st.u_tok = ut;
    if (ab == Lb) {
        // Bonus draw from p of row L_b: block masses from the tile records.
        const float4 *rec = a.rec + size_t(r0 + Lb) * a.nblk_stride;
        auto mass = [&](int i) {
            const float4 x = __ldcg(rec + i);
            return x.y > 0.f ? x.y * exp2_approx((x.x - Mbonus) * scale) : 0.f;
        };
        const int blk = choose_block(nb, ub, mass, lane);
        st.mode = D_BONUS;
        st.Mp = Mbonus;
        st.Sp = 1.f;
        st.Mq = 0.f;
        st.Sq = 1.f;
        if (lane == 0) {
            a.dstate[b] = st;
            push_jobs(a, T_PICK, b, blk, 1, epoch);
        }
    } else {
        st.mode = D_RESID;
        st.Mp = Mp;
        st.Sp = Sp;
        st.Mq = Mq;
        st.Sq = Sq;
        if (lane == 0) {
            a.dstate[b] = st;
            push_jobs(a, T_RESID, b, 0, a.nc, epoch);
        }
    }
}

// All residual-mass tiles of request b are in: choose the block (warp-level).
__device__ void decide_residual_block(const VerifyArgs &a, int b, int epoch, int lane) {
    DecideState st = load_state(a, b);
    const float *z = a.zrec + size_t(b) * a.nblk_stride;
    double total = 0.0;
    for (int t0 = 0; t0 < a.nblk; t0 += 32) {
        const int i = t0 + lane;
        double v = i < a.nblk ? double(__ldcg(z + i)) : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        total += v;
    }
    int blk;
    if (total > 0.0) {
        blk = choose_block(a.nblk, st.u_blk, [&](int i) { return __ldcg(z + i); }, lane);
    } else {
        // No residual mass: draw from p of the same row instead.
        const float4 *rec = a.rec + size_t(a.row_off[b] + st.a) * a.nblk_stride;
        const float M = st.Mp, scale = a.scale;
        blk = choose_block(a.nblk, st.u_blk, [&](int i) {
            const float4 x = __ldcg(rec + i);
            return x.y > 0.f ? x.y * exp2_approx((x.x - M) * scale) : 0.f;
        }, lane);
        st.mode = D_FALLBACK;
        st.Sp = 1.f;
    }
    if (lane == 0) {
        a.dstate[b] = st;
        push_jobs(a, T_PICK, b, blk, 1, epoch);
    }
}

// ---------------------------------------------------------------------------
// consumers
// ---------------------------------------------------------------------------
// Draw weights of the VE elements of 16-byte vector v: 2^((z - Mp) s) for a
// draw from p (bonus, fallback); max(0, p - q) for the residual.
template <typename T>
__device__ __forceinline__ void draw_weights(const uint4 *tv, const uint4 *dv, int v, int mode,
                                             float Mp, float iSp, float Mq, float iSq,
                                             float scale, float (&w)[Vec<T>::kElems]) {
    constexpr int VE = Vec<T>::kElems;
    float x[VE];
    Vec<T>::unpack(tv[v], x);
    if (mode == D_RESID) {
        float y[VE];
        Vec<T>::unpack(dv[v], y);
#pragma unroll
        for (int e = 0; e < VE; ++e)
            w[e] = fmaxf(0.f, exp2_approx((x[e] - Mp) * scale) * iSp -
                                  exp2_approx((y[e] - Mq) * scale) * iSq);
    } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) w[e] = exp2_approx((x[e] - Mp) * scale);
    }
}

// Sum of the draw weights of a lane's contiguous run [v0, v0 + per).
template <typename T>
__device__ __forceinline__ float run_weight(const uint4 *tv, const uint4 *dv, int v0, int per,
                                            int nvec, const DecideState &st, float iSp,
                                            float iSq, float scale) {
    constexpr int VE = Vec<T>::kElems;
    float ls = 0.f;
    for (int q = 0; q < per; ++q) {
        const int v = v0 + q;
        if (v < nvec) {
            float w[VE];
            draw_weights<T>(tv, dv, v, st.mode, st.Mp, iSp, st.Mq, iSq, scale, w);
#pragma unroll
            for (int e = 0; e < VE; ++e) ls += w[e];
        }
    }
    return ls;
}

// The pick of a stage holding one sampling block (warp-level, by the
// stage's last warp): the warp share, then the lane run, then the token.
template <typename T>
__device__ int pick_token(const VSmem &sm, int s, const TaskInfo &t, const DecideState &st,
                          const uint4 *tv, const uint4 *dv, float scale, int lane) {
    constexpr int VE = Vec<T>::kElems;
    const int nvec = t.bytes / 16;
    const double wv = lane < kCW ? sm.wd[s][lane] : 0.0;
    const double wincl = warp_scan_incl(wv, lane);
    const double total = __shfl_sync(0xffffffffu, wincl, kCW - 1);
    const double target = double(st.u_tok) * total;
    unsigned hit = __ballot_sync(0xffffffffu, lane < kCW && wincl > target);
    const unsigned posw = __ballot_sync(0xffffffffu, lane < kCW && wv > 0.0);
    const int ws = hit ? __ffs(hit) - 1 : (posw ? 31 - __clz(posw) : 0);
    const double wprev = __shfl_sync(0xffffffffu, wincl, ws > 0 ? ws - 1 : 0);
    const double wbase = ws > 0 ? wprev : 0.0;
    const float iSp = 1.f / st.Sp, iSq = 1.f / st.Sq;
    const int pv = kSampleBlock / VE / kCW;  // vectors per warp share
    const int per = pv / 32;                 // vectors per lane run
    const int v0 = ws * pv + lane * per;
    const float ls = run_weight<T>(tv, dv, v0, per, nvec, st, iSp, iSq, scale);
    const double lincl = warp_scan_incl(double(ls), lane);
    const double lprev = __shfl_up_sync(0xffffffffu, lincl, 1);
    const double lexcl = lane > 0 ? lprev : 0.0;
    hit = __ballot_sync(0xffffffffu, ls > 0.f && wbase + lincl > target);
    const unsigned posl = __ballot_sync(0xffffffffu, ls > 0.f);
    const int lsel = hit ? __ffs(hit) - 1 : (posl ? 31 - __clz(posl) : -1);
    if (lsel < 0) return t.y0 + ws * pv * VE;  // the whole share carries no weight
    int pick = -1;
    if (lane == lsel) {
        int lastpos = -1;
        float run = 0.f;
        for (int q = 0; q < per && pick < 0; ++q) {
            const int v = v0 + q;
            if (v >= nvec) break;
            float w[VE];
            draw_weights<T>(tv, dv, v, st.mode, st.Mp, iSp, st.Mq, iSq, scale, w);
#pragma unroll
            for (int e = 0; e < VE; ++e) {
                run += w[e];
                if (pick < 0 && w[e] > 0.f) {
                    lastpos = v * VE + e;
                    if (wbase + lexcl + double(run) > target) pick = v * VE + e;
                }
            }
        }
        if (pick < 0) pick = lastpos;
    }
    return t.y0 + __shfl_sync(0xffffffffu, pick, lsel);
}

template <typename T>
__device__ void consumer(const VerifyArgs &a, VSmem &sm, const uint8_t *ring, int warp, int lane,
                         int epoch) {
    constexpr int VE = Vec<T>::kElems;
    const float scale = a.scale;
    const int tpw = a.chunk_elems / kCW;  // tokens per warp in a tile
    const int vpw = tpw / VE;             // vectors per warp in a tile
    const int wpb = kSampleBlock / tpw;   // warps per sampling block
    const int bpc = kCW / wpb;            // sampling blocks per tile
    for (int fill = 0;; ++fill) {
        const int s = fill % kStages, n = fill / kStages;
        if (!mbar_wait_bounded(&sm.full[s], n & 1)) {
            if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
            return;
        }
        const TaskInfo t = sm.task[s];
        if (t.type == T_EXIT) return;
        const uint4 *tv = reinterpret_cast<const uint4 *>(ring + s * kStageBytes);
        const uint4 *dv = tv + kChunkBytes / 16;
        const int nvec = t.bytes / 16;

        if (t.type == T_STREAM) {
            const int v0 = min(nvec, warp * vpw), v1 = min(nvec, v0 + vpw);
            if (a.greedy) {
                float bv = -INFINITY;
                int bi = INT_MAX;
                for (int v = v0 + lane; v < v1; v += 32) {
                    float z[VE];
                    Vec<T>::unpack(tv[v], z);
#pragma unroll
                    for (int e = 0; e < VE; ++e)
                        if (z[e] > bv) {
                            bv = z[e];
                            bi = t.y0 + v * VE + e;
                        }
                }
                warp_am_reduce(bv, bi);
                if (lane == 0) sm.wpart[s][warp] = make_float4(bv, __int_as_float(bi), 0.f, 0.f);
            } else {
                float mp = -INFINITY, sp = 0.f, mq = -INFINITY, sq = 0.f;
                if (t.pair) {
                    for (int v = v0 + lane; v < v1; v += 32) {
                        float z[VE];
                        Vec<T>::unpack(tv[v], z);
                        online_update<VE>(mp, sp, z, scale);
                        Vec<T>::unpack(dv[v], z);
                        online_update<VE>(mq, sq, z, scale);
                    }
                    warp_ms_reduce(mq, sq, scale);
                } else {
                    for (int v = v0 + lane; v < v1; v += 32) {
                        float z[VE];
                        Vec<T>::unpack(tv[v], z);
                        online_update<VE>(mp, sp, z, scale);
                    }
                }
                warp_ms_reduce(mp, sp, scale);
                if (lane == 0) {
                    sm.wpart[s][warp] = make_float4(mp, sp, mq, sq);
                    if (t.pair) {
                        const int dt = t.d;
                        const int lo = t.y0 + v0 * VE, hi = t.y0 + v1 * VE;
                        if (dt >= lo && dt < hi) {
                            sm.gath[s] = make_float2(Vec<T>::load1(tv, dt - t.y0),
                                                     Vec<T>::load1(dv, dt - t.y0));
                            sm.gflag[s] = 1;
                        }
                    }
                }
            }
        } else if (t.type == T_RESID) {
            const DecideState st = load_state(a, t.b);
            const float iSp = 1.f / st.Sp, iSq = 1.f / st.Sq;
            const int v0 = min(nvec, warp * vpw), v1 = min(nvec, v0 + vpw);
            float zs = 0.f;
            for (int v = v0 + lane; v < v1; v += 32) {
                float w[VE];
                draw_weights<T>(tv, dv, v, D_RESID, st.Mp, iSp, st.Mq, iSq, scale, w);
#pragma unroll
                for (int e = 0; e < VE; ++e) zs += w[e];
            }
            double zd = zs;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) zd += __shfl_xor_sync(0xffffffffu, zd, o);
            if (lane == 0) sm.wd[s][warp] = zd;
        } else if (t.type == T_PICK) {  // each lane sums one contiguous run of its warp's share
            const DecideState st = load_state(a, t.b);
            const float iSp = 1.f / st.Sp, iSq = 1.f / st.Sq;
            const int pv = kSampleBlock / VE / kCW;
            const int per = pv / 32;
            const float ls = run_weight<T>(tv, dv, warp * pv + lane * per, per, nvec, st, iSp,
                                           iSq, scale);
            const double incl = warp_scan_incl(double(ls), lane);
            if (lane == 31) sm.wd[s][warp] = incl;
        }

        // Elect the stage's last warp; it finishes the stage.
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&sm.done[s], 1) == kCW - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence_block();
            if (lane == 0) sm.done[s] = 0;
            if (t.type == T_STREAM) {
                const int blk0 = t.j * bpc;
                if (lane < bpc && blk0 + lane < a.nblk) {
                    float4 r;
                    if (a.greedy) {
                        float bv = -INFINITY;
                        int bi = INT_MAX;
                        for (int w = lane * wpb; w < (lane + 1) * wpb; ++w)
                            am_combine(bv, bi, sm.wpart[s][w].x, __float_as_int(sm.wpart[s][w].y));
                        r = make_float4(bv, __int_as_float(bi), 0.f, 0.f);
                    } else {
                        float mp = -INFINITY, sp = 0.f, mq = -INFINITY, sq = 0.f;
                        for (int w = lane * wpb; w < (lane + 1) * wpb; ++w) {
                            const float4 x = sm.wpart[s][w];
                            ms_combine(mp, sp, x.x, x.y, scale);
                            ms_combine(mq, sq, x.z, x.w, scale);
                        }
                        r = make_float4(mp, sp, mq, sq);
                    }
                    a.rec[size_t(t.r) * a.nblk_stride + blk0 + lane] = r;
                }
                if (lane == 0 && sm.gflag[s]) {
                    a.gath[t.r] = sm.gath[s];
                    sm.gflag[s] = 0;
                }
            } else if (t.type == T_RESID) {
                const int blk0 = t.j * bpc;
                if (lane < bpc && blk0 + lane < a.nblk) {
                    double z = 0.0;
                    for (int w = lane * wpb; w < (lane + 1) * wpb; ++w) z += sm.wd[s][w];
                    a.zrec[size_t(t.b) * a.nblk_stride + blk0 + lane] = float(z);
                }
            } else if (t.type == T_PICK) {
                const DecideState st = load_state(a, t.b);
                const int token = pick_token<T>(sm, s, t, st, tv, dv, scale, lane);
                finish_request(a, t.b, st.a, token, lane);
            } else if (t.type == T_DECIDE) {
                __threadfence();
                decide_request(a, t.b, epoch, lane);
            } else {
                __threadfence();
                decide_residual_block(a, t.b, epoch, lane);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);
    }
}

template <typename T>
__global__ void __launch_bounds__(kVerifyThreads, 2) verify_kernel(const VerifyArgs a) {
    extern __shared__ __align__(1024) uint8_t ring[];
    __shared__ VSmem sm;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int epoch = a.q_ctr[Q_EPOCH] + 1;
    if (tid < kStages) {
        mbar_init(&sm.full[tid], 1);
        mbar_init(&sm.empty[tid], kCW);
        sm.done[tid] = 0;
        sm.gflag[tid] = 0;
    }
    if (tid == 0) fence_barrier_init();
    __syncthreads();

    // Packed rows as written by the compaction, never more than its capacity.
    const int n_rows = min(max(a.row_off[a.B], 0), a.B * (a.gamma + 1));
    const long long n_tasks = (long long)n_rows * a.nc;
    const long long G = gridDim.x;
    const long long s_lo = n_tasks * blockIdx.x / G, s_hi = n_tasks * (blockIdx.x + 1) / G;

    if (warp == kCW) {
        if (lane == 0) producer(a, sm, ring, s_lo, s_hi, n_rows, epoch);
    } else {
        consumer<T>(a, sm, ring, warp, lane, epoch);
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(&a.q_ctr[Q_EXITED], 1) == int(G) - 1) {
            // Every CTA is done: reset the queue for the next launch.
            a.q_ctr[Q_HEAD] = 0;
            a.q_ctr[Q_TAIL] = 0;
            a.q_ctr[Q_FINISHED] = 0;
            a.q_ctr[Q_EXITED] = 0;
            a.q_ctr[Q_EPOCH] = epoch;
            __threadfence();
        }
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
    // Cooperative launch: the producers poll a device-wide queue, so every
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
