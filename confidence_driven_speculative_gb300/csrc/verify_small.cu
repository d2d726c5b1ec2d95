// verify_small.cu -- steps a5-a6 for small batches, with no queue and no
// persistent roles.
//
// Same method as verify.cu ("DFlash to DSpark in SGLang", section
// "Background"; "SGLang Integrates DSpark ...", section "The Old Problem with
// Speculative Decoding": accept draft d with probability min(1, p(d)/q(d)),
// on the first rejection draw from norm(max(0, p - q)), else the bonus token
// from p at row L_b), and the same two-level draw over 4096-id blocks with
// the uniforms (u, u', u'') of Philox words 0, 1, 2 at counter (b, k).
//
// Design (GB300, small B).  With few rows the large kernel's cost is its
// chains of queue hops, not bytes.  Here a grid of plain CTAs takes units
// (packed row r, slice j of 8192 ids) in a fixed stride, no atomics: a unit
// reads its slice of the target row and, for a decision row, of the draft
// row with 16-byte vector loads and writes the slice's record -- online
// (max, sum of 2^(z s - max)) of p and q, the greedy argmax (lowest id on
// ties), or for a bonus row the (max, sum) of each 4096-id block -- and the
// drafted id's two logits when they fall in the slice.  It then counts the
// unit towards its request; the CTA that completes the request's units
// decides it with all 256 threads: accept tests from the row records, then
// the residual draw (it streams the rejected row pair once more, block masses
// per warp, in two-float sums) or the bonus draw from the bonus row's block
// records, each a block by u' and an id inside it by u''.  With rows of four
// tiles or more and four requests or more (small_tail), a rejection is listed
// instead for the tail kernel
// (verify.cu), which takes the row pair's second pass in parts over the
// whole GPU and makes the residual draw: one CTA alone needs ~25 us for a
// 300 KB row pair, a second launch a few us.
//
// Waits: none.  Every CTA runs to completion on its own units.
#include <climits>

#include "dspark_internal.cuh"

namespace dspark {
namespace {

constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSliceIds = 8192;  // token ids per unit (two sampling blocks)
static_assert(kSliceIds % kSampleBlock == 0, "a slice holds whole sampling blocks");
constexpr int kBlkPerSlice = kSliceIds / kSampleBlock;
constexpr int kMaxBlocks = 64;  // sampling blocks of a row this path takes (V <= 262144)

// Two-float numbers (hi + lo): sums of fp32 masses as exact as fp64 (Knuth's
// TwoSum keeps each addition's rounding error) on the fp32 pipe.
struct F2s {
    float hi, lo;
};
__device__ __forceinline__ F2s f2s(float x) { return F2s{x, 0.f}; }
__device__ __forceinline__ F2s add(F2s a, F2s b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    const float e = (a.hi - (s - bb)) + (b.hi - bb) + (a.lo + b.lo);
    const float h = s + e;
    return F2s{h, e - (h - s)};
}
__device__ __forceinline__ F2s scale_by(F2s a, float u) {  // a * u, 0 <= u <= 1
    const float p = a.hi * u;
    const float e = fmaf(a.hi, u, -p) + a.lo * u;
    const float h = p + e;
    return F2s{h, e - (h - p)};
}
__device__ __forceinline__ bool gt(F2s a, F2s b) { return (a.hi - b.hi) + (a.lo - b.lo) > 0.f; }
__device__ __forceinline__ F2s shfl_xor(F2s v, int o) {
    return F2s{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ F2s shfl_up(F2s v, int o) {
    return F2s{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ F2s warp_sum(F2s v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = add(v, shfl_xor(v, o));
    return v;
}

template <int VE>
__device__ __forceinline__ void online(float &m, float &s, const float (&x)[VE], float scale) {
    float vm = x[0];
#pragma unroll
    for (int e = 1; e < VE; ++e) vm = fmaxf(vm, x[e]);
    if (vm > m) {
        s *= exp2_approx((m - vm) * scale);
        m = vm;
    }
    const float ms = m * scale;
    float t = 0.f;
#pragma unroll
    for (int e = 0; e < VE; ++e) t += exp2_approx(fmaf(x[e], scale, -ms));
    s += t;
}

struct SmallSmem {
    float4 red[kSmallWarps];          // warp partials of a unit
    int last;                         // this CTA completed the request
    // decision of a request
    float4 norm[DSPARK_MAX_GAMMA + 1];  // (Mp, Sp, Mq, Sq) per decision row
    int acc[DSPARK_MAX_GAMMA];        // accept test of each draft
    int gtok[DSPARK_MAX_GAMMA + 1];   // greedy argmax of each row
    float2 blk[kMaxBlocks];           // block masses of a draw (hi, lo)
    float2 thr[kSmallThreads];        // per-thread partial sums of the in-block scan
    int pick;                         // chosen block / id
};

// CTA-wide combine of per-thread (max, sum) pairs (two of them in a float4)
// or (value, index) argmax pairs; the result lands in every thread.
__device__ float4 cta_ms(SmallSmem &sm, float4 x, float scale, bool greedy) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (greedy) {
        int i = __float_as_int(x.y);
        warp_am_reduce(x.x, i);
        x.y = __int_as_float(i);
    } else {
        warp_ms_reduce(x.x, x.y, scale);
        warp_ms_reduce(x.z, x.w, scale);
    }
    __syncthreads();
    if (lane == 0) sm.red[warp] = x;
    __syncthreads();
    float4 y = sm.red[0];
    for (int w = 1; w < kSmallWarps; ++w) {
        const float4 z = sm.red[w];
        if (greedy) {
            int i = __float_as_int(y.y);
            am_combine(y.x, i, z.x, __float_as_int(z.y));
            y.y = __int_as_float(i);
        } else {
            ms_combine(y.x, y.y, z.x, z.y, scale);
            ms_combine(y.z, y.w, z.z, z.w, scale);
        }
    }
    return y;
}

// One unit: slice j of packed row r (request b, draft index k, verify length
// Lb).  Writes the slice's record and, for a decision row, the drafted id's
// logits if the slice holds it.
template <typename T>
__device__ void run_unit(const VerifyArgs &a, SmallSmem &sm, int r, int j, int b, int k, int Lb) {
    constexpr int VE = Vec<T>::kElems;
    const int tid = threadIdx.x;
    const float scale = a.scale;
    const int y0 = j * kSliceIds, y1 = min(a.V, y0 + kSliceIds);
    const int v0 = y0 / VE, v1 = (y1 + VE - 1) / VE;  // V * elem is a multiple of 16 bytes
    const uint4 *tv = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.target_logits) +
                                                      size_t(r) * a.row_bytes);
    if (a.greedy) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        constexpr int kPer = kSliceIds / VE / kSmallThreads;
        uint4 xt[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int v = v0 + tid + i * kSmallThreads;
            xt[i] = v < v1 ? __ldg(tv + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int v = v0 + tid + i * kSmallThreads;
            if (v >= v1) continue;
            float z[VE];
            Vec<T>::unpack(xt[i], z);
#pragma unroll
            for (int e = 0; e < VE; ++e)
                if (z[e] > bv) {
                    bv = z[e];
                    bi = v * VE + e;
                }
        }
        const float4 y = cta_ms(sm, make_float4(bv, __int_as_float(bi), 0.f, 0.f), scale, true);
        if (tid == 0) a.rowrec[size_t(r) * a.grp_stride + j] = y;
        return;
    }
    if (k < Lb) {
        const uint4 *dv = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.draft_logits) +
                                                          (size_t(b) * a.gamma + k) * a.row_bytes);
        float mp = -INFINITY, sp = 0.f, mq = -INFINITY, sq = 0.f;
        // every load of the thread is issued before the first is used
        constexpr int kPer = kSliceIds / VE / kSmallThreads;
        uint4 xt[kPer], xd[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int v = v0 + tid + i * kSmallThreads;
            xt[i] = v < v1 ? __ldg(tv + v) : make_uint4(0, 0, 0, 0);
            xd[i] = v < v1 ? __ldg(dv + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            if (v0 + tid + i * kSmallThreads >= v1) continue;
            float z[VE];
            Vec<T>::unpack(xt[i], z);
            online<VE>(mp, sp, z, scale);
            Vec<T>::unpack(xd[i], z);
            online<VE>(mq, sq, z, scale);
        }
        const float4 y = cta_ms(sm, make_float4(mp, sp, mq, sq), scale, false);
        if (tid == 0) {
            a.rowrec[size_t(r) * a.grp_stride + j] = y;
            const int d = a.draft_tokens[size_t(b) * a.gamma + k];
            if (d >= y0 && d < y1)
                a.gath[r] = make_float2(Vec<T>::load1(tv, d), Vec<T>::load1(dv, d));
        }
        return;
    }
    // Bonus row: (max, sum) of each 4096-id block of the slice, one warp
    // group of 128 threads per block.
    const int half = tid / (kSmallThreads / kBlkPerSlice);
    const int t2 = tid % (kSmallThreads / kBlkPerSlice);
    const int by0 = y0 + half * kSampleBlock, by1 = min(y1, by0 + kSampleBlock);
    float m = -INFINITY, sum = 0.f;
    {
        constexpr int kStep = kSmallThreads / kBlkPerSlice;
        constexpr int kPer = kSampleBlock / VE / kStep;
        const int va = by0 / VE + t2, vb = (by1 + VE - 1) / VE;
        uint4 xb[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            xb[i] = va + i * kStep < vb ? __ldg(tv + va + i * kStep) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            if (va + i * kStep >= vb) continue;
            float z[VE];
            Vec<T>::unpack(xb[i], z);
            online<VE>(m, sum, z, scale);
        }
    }
    const int lane = tid & 31, warp = tid >> 5;
    warp_ms_reduce(m, sum, scale);
    __syncthreads();
    if (lane == 0) sm.red[warp] = make_float4(m, sum, 0.f, 0.f);
    __syncthreads();
    if (tid < kBlkPerSlice) {
        const int wpb = kSmallWarps / kBlkPerSlice;
        float4 acc4 = sm.red[tid * wpb];
        for (int w = 1; w < wpb; ++w) ms_combine(acc4.x, acc4.y, sm.red[tid * wpb + w].x,
                                                 sm.red[tid * wpb + w].y, scale);
        const int blk = y0 / kSampleBlock + tid;
        if (blk < a.nblk && y0 + tid * kSampleBlock < a.V)
            a.blkrec[(size_t(b) * a.nblk + blk) * kConsumerWarps] = make_float2(acc4.x, acc4.y);
    }
}

// Weight of id y in a draw: the residual max(0, p - q) (normalised by the
// rows' (M, S)), or p's unnormalised 2^((z - M) s).
struct DrawRows {
    const uint4 *tv, *dv;  // target and draft rows (dv: residual only)
    bool resid;
    float Mp, iSp, Mq, iSq, scale;
};

template <typename T>
__device__ __forceinline__ void weights(const DrawRows &w, int v, float (&out)[Vec<T>::kElems]) {
    constexpr int VE = Vec<T>::kElems;
    float x[VE];
    Vec<T>::unpack(__ldg(w.tv + v), x);
    if (w.resid) {
        float y[VE];
        Vec<T>::unpack(__ldg(w.dv + v), y);
#pragma unroll
        for (int e = 0; e < VE; ++e)
            out[e] = fmaxf(0.f, exp2_approx((x[e] - w.Mp) * w.scale) * w.iSp -
                                    exp2_approx((y[e] - w.Mq) * w.scale) * w.iSq);
    } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) out[e] = exp2_approx((x[e] - w.Mp) * w.scale);
    }
}

// Masses of every sampling block of the draw's row (warp w takes blocks w,
// w + 8, ...), into sm.blk; returns their total (every thread).
template <typename T>
__device__ F2s block_masses(const VerifyArgs &a, SmallSmem &sm, const DrawRows &w) {
    constexpr int VE = Vec<T>::kElems;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int vend = a.V / VE;
    for (int blk = warp; blk < a.nblk; blk += kSmallWarps) {
        const int vb = blk * (kSampleBlock / VE);
        F2s m = f2s(0.f);
        const int ve = min(vend, vb + kSampleBlock / VE);
        constexpr int kBatch = 8;  // vectors per lane in flight
        for (int v = vb + lane; v < ve; v += 32 * kBatch) {
            float t[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                t[i] = 0.f;
                if (v + 32 * i < ve) {
                    float wt[VE];
                    weights<T>(w, v + 32 * i, wt);
#pragma unroll
                    for (int e = 0; e < VE; ++e) t[i] += wt[e];
                }
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i) m = add(m, f2s(t[i]));
        }
        m = warp_sum(m);
        if (lane == 0) sm.blk[blk] = make_float2(m.hi, m.lo);
    }
    __syncthreads();
    F2s z = f2s(0.f);
    for (int i = 0; i < a.nblk; ++i) z = add(z, F2s{sm.blk[i].x, sm.blk[i].y});
    return z;
}

// The two-level draw from the masses in sm.blk (total Z): the smallest block
// whose running mass exceeds u' Z, then the smallest id in it whose running
// weight exceeds u'' times the block's mass; rounding fallbacks: the last
// block / id with positive weight.  Returns the id (every thread).
template <typename T>
__device__ int draw_two_level(const VerifyArgs &a, SmallSmem &sm, const DrawRows &w, F2s Z,
                              float u_blk, float u_tok) {
    constexpr int VE = Vec<T>::kElems;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        const F2s t = scale_by(Z, u_blk);
        F2s run = f2s(0.f);
        int pick = -1, lastpos = 0;
        for (int i = 0; i < a.nblk && pick < 0; ++i) {
            const F2s m = F2s{sm.blk[i].x, sm.blk[i].y};
            if (m.hi > 0.f) lastpos = i;
            run = add(run, m);
            if (m.hi > 0.f && gt(run, t)) pick = i;
        }
        sm.pick = pick >= 0 ? pick : lastpos;
    }
    __syncthreads();
    const int blk = sm.pick;
    // In-block: thread t owns ids blk*4096 + 16t .. +16 (two or four vectors).
    constexpr int kPer = kSampleBlock / kSmallThreads;  // 16 ids per thread
    constexpr int kVec = kPer / VE;
    const int vbase = (blk * kSampleBlock + tid * kPer) / VE;
    const int vend = a.V / VE;
    float wt[kVec][VE];
    float part = 0.f;
#pragma unroll
    for (int q = 0; q < kVec; ++q) {
        if (vbase + q < vend) {
            weights<T>(w, vbase + q, wt[q]);
        } else {
#pragma unroll
            for (int e = 0; e < VE; ++e) wt[q][e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) part += wt[q][e];
    }
    // exclusive scan of the 256 parts in two-float sums
    F2s incl = f2s(part);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const F2s n = shfl_up(incl, o);
        if (lane >= o) incl = add(incl, n);
    }
    if (lane == 31) sm.thr[warp] = make_float2(incl.hi, incl.lo);
    __syncthreads();
    F2s before = f2s(0.f), mass = f2s(0.f);
    for (int i = 0; i < kSmallWarps; ++i) {
        const F2s x = F2s{sm.thr[i].x, sm.thr[i].y};
        if (i < warp) before = add(before, x);
        mass = add(mass, x);
    }
    const F2s excl = add(before, add(incl, F2s{-part, 0.f}));
    const F2s t2 = scale_by(mass, u_tok);
    __syncthreads();
    if (tid == 0) sm.pick = -1;
    __syncthreads();
    // the thread whose run crosses t2 finds the id
    const F2s end = add(before, incl);
    if (part > 0.f && gt(end, t2) && !gt(excl, t2) ) {
        F2s run = excl;
        int id = -1, lastpos = -1;
#pragma unroll
        for (int q = 0; q < kVec; ++q)
#pragma unroll
            for (int e = 0; e < VE; ++e) {
                if (id < 0 && wt[q][e] > 0.f) {
                    lastpos = (vbase + q) * VE + e;
                    run = add(run, f2s(wt[q][e]));
                    if (gt(run, t2)) id = (vbase + q) * VE + e;
                }
            }
        atomicMax(&sm.pick, id >= 0 ? id : lastpos);
    }
    __syncthreads();
    int id = sm.pick;
    if (id < 0) {
        // rounding left no crossing: the last id with positive weight
        int lp = -1;
#pragma unroll
        for (int q = 0; q < kVec; ++q)
#pragma unroll
            for (int e = 0; e < VE; ++e)
                if (wt[q][e] > 0.f) lp = (vbase + q) * VE + e;
        __syncthreads();
        atomicMax(&sm.pick, lp);
        __syncthreads();
        id = sm.pick >= 0 ? sm.pick : blk * kSampleBlock;
    }
    __syncthreads();
    return id;
}

// Request b's units are all in: decide it and emit (all 256 threads).
template <typename T>
__device__ void finish_request_small(const VerifyArgs &a, SmallSmem &sm, int b, int S) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float scale = a.scale;
    const int Lb = min(max(a.L[b], 0), a.gamma);
    const int r0 = a.row_off[b], d0 = a.draft_off[b];
    const int32_t *drafts = a.draft_tokens + size_t(b) * a.gamma;
    // Row records: warp w takes rows w, w + 8, ... (decision rows; greedy
    // also the bonus row), lane j record j.
    const int rows = a.greedy ? Lb + 1 : Lb;
    for (int k = warp; k < rows; k += kSmallWarps) {
        const float4 *rec = a.rowrec + size_t(r0 + k) * a.grp_stride;
        float4 x = a.greedy ? make_float4(-INFINITY, __int_as_float(INT_MAX), 0.f, 0.f)
                            : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        for (int j = lane; j < S; j += 32) {
            const float4 y = __ldcg(rec + j);
            if (a.greedy) {
                int i = __float_as_int(x.y);
                am_combine(x.x, i, y.x, __float_as_int(y.y));
                x.y = __int_as_float(i);
            } else {
                ms_combine(x.x, x.y, y.x, y.y, scale);
                ms_combine(x.z, x.w, y.z, y.w, scale);
            }
        }
        if (a.greedy) {
            int i = __float_as_int(x.y);
            warp_am_reduce(x.x, i);
            if (lane == 0) {
                sm.gtok[k] = i;
                if (k < Lb) {
                    sm.acc[k] = drafts[k] == i;
                    a.p_tok[d0 + k] = 0.f;
                    a.q_tok[d0 + k] = 0.f;
                }
            }
        } else {
            warp_ms_reduce(x.x, x.y, scale);
            warp_ms_reduce(x.z, x.w, scale);
            if (lane == 0) {
                sm.norm[k] = x;
                const int d = drafts[k];
                float p = 0.f, q = 0.f, ratio = 0.f;
                if (d >= 0 && d < a.V) {
                    const float2 z = __ldcg(a.gath + r0 + k);
                    p = exp2_approx((z.x - x.x) * scale) / x.y;
                    q = exp2_approx((z.y - x.z) * scale) / x.w;
                    ratio = q > 0.f ? fminf(1.f, p / q) : 1.f;
                }
                float u, u1, u2;
                step_uniforms(a.seed, b, k, u, u1, u2);
                sm.acc[k] = u < ratio;
                a.p_tok[d0 + k] = p;
                a.q_tok[d0 + k] = q;
            }
        }
    }
    __syncthreads();
    int acc = Lb;
    for (int k = 0; k < Lb; ++k)
        if (!sm.acc[k]) {
            acc = k;
            break;
        }
    int token;
    if (a.greedy) {
        token = sm.gtok[acc];
    } else {
        float u, u_blk, u_tok;
        step_uniforms(a.seed, b, acc, u, u_blk, u_tok);
        DrawRows w;
        w.scale = scale;
        if (acc < Lb && a.small_tail) {
            // The residual at row acc (from p if its mass is zero) is the tail
            // kernel's: listed with the row and the draw state, the row's
            // second pass is cut into parts over the whole GPU there (one CTA
            // alone took ~25 us for a 300 KB row pair).  It writes the outputs.
            if (tid == 0) {
                const float4 nm = sm.norm[acc];
                DecideState st;
                st.a = acc;
                st.mode = D_RESID;
                st.Mp = nm.x;
                st.Sp = nm.y;
                st.Mq = nm.z;
                st.Sq = nm.w;
                st.u_blk = u_blk;
                st.u_tok = u_tok;
                const int pos = atomicAdd(&a.q_ctr[kQSmallList], 1);  // each request once: < B
                if (pos < a.B) {
                    a.q_job[pos] = make_int2(b, r0 + acc);
                    a.dstate[pos] = st;
                }
                a.req_cnt[b] = 0;  // complete here: reset for the next launch
            }
            return;
        }
        if (acc < Lb) {
            // residual at row acc, from p if its mass is zero (rows of a few
            // tiles: one CTA's pass costs less than a second launch)
            const float4 nm = sm.norm[acc];
            w.tv = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.target_logits) +
                                                   size_t(r0 + acc) * a.row_bytes);
            w.dv = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.draft_logits) +
                                                   (size_t(b) * a.gamma + acc) * a.row_bytes);
            w.resid = true;
            w.Mp = nm.x;
            w.iSp = 1.f / nm.y;
            w.Mq = nm.z;
            w.iSq = 1.f / nm.w;
            F2s Z = block_masses<T>(a, sm, w);
            if (!(Z.hi > 0.f)) {
                __syncthreads();
                w.resid = false;
                Z = block_masses<T>(a, sm, w);
            }
            token = draw_two_level<T>(a, sm, w, Z, u_blk, u_tok);
        } else {
            // bonus: p at row L_b from its block records
            const float2 *rec = a.blkrec + size_t(b) * a.nblk * kConsumerWarps;
            if (tid < a.nblk) {
                const float2 x = __ldcg(rec + size_t(tid) * kConsumerWarps);
                sm.thr[tid] = x;
            }
            __syncthreads();
            float M = -INFINITY;
            for (int i = 0; i < a.nblk; ++i)
                if (sm.thr[i].y > 0.f) M = fmaxf(M, sm.thr[i].x);
            __syncthreads();
            if (tid < a.nblk) {
                const float2 x = sm.thr[tid];
                sm.blk[tid] = make_float2(x.y > 0.f ? x.y * exp2_approx((x.x - M) * scale) : 0.f, 0.f);
            }
            __syncthreads();
            F2s Z = f2s(0.f);
            for (int i = 0; i < a.nblk; ++i) Z = add(Z, F2s{sm.blk[i].x, sm.blk[i].y});
            w.tv = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.target_logits) +
                                                   size_t(r0 + Lb) * a.row_bytes);
            w.dv = w.tv;
            w.resid = false;
            w.Mp = M;
            w.iSp = w.Mq = w.iSq = 1.f;
            token = draw_two_level<T>(a, sm, w, Z, u_blk, u_tok);
        }
    }
    // outputs
    const int g1 = a.gamma + 1;
    for (int j = tid; j < g1; j += kSmallThreads) {
        int v = -1;
        if (j < acc) v = drafts[j];
        else if (j == acc) v = token;
        a.out_tokens[size_t(b) * g1 + j] = v;
    }
    if (tid == 0) {
        a.accept_len[b] = acc;
        a.num_emitted[b] = acc + 1;
        if (a.seq_lens_commit) a.seq_lens_commit[b] += acc + 1;
        a.req_cnt[b] = 0;  // complete: reset for the next launch
    }
}

template <typename T>
__global__ void __launch_bounds__(kSmallThreads) verify_small_kernel(const VerifyArgs a, int S) {
    // Launched as a programmatic dependent of the kernel before it: wait for
    // it.  The tail kernel after it may be scheduled as this grid's CTAs
    // leave (it waits for this grid to complete).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ SmallSmem sm;
    const int tid = threadIdx.x;
    const int cap = a.B * (a.gamma + 1);
    // The first unit's row ids go out with the packed total (the row-id
    // arrays hold the batch's capacity): one round trip less before its data.
    const int r_first = int(blockIdx.x) / S;
    const int b_first = r_first < cap ? a.row_req[r_first] : 0;
    const int k_first = r_first < cap ? a.row_k[r_first] : 0;
    const int n_rows = min(max(a.row_off[a.B], 0), cap);
    const int units = n_rows * S;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int r = u / S, j = u - r * S;
        const bool first = u == int(blockIdx.x);
        const int b = min(max(first ? b_first : a.row_req[r], 0), a.B - 1);
        const int k = max(first ? k_first : a.row_k[r], 0);
        // Greedy units read the target row only: L_b's load (needed for the
        // count) goes out beside theirs instead of before them.
        const int L_raw = a.L[b];
        const int Lb = a.greedy ? 0 : min(max(L_raw, 0), a.gamma);
        run_unit<T>(a, sm, r, j, b, k, Lb);
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            sm.last = atomicAdd(&a.req_cnt[b], 1) == (min(max(L_raw, 0), a.gamma) + 1) * S - 1;
        }
        __syncthreads();
        if (sm.last) {
            __threadfence();
            finish_request_small<T>(a, sm, b, S);
        }
        __syncthreads();
    }
}

}  // namespace

// Slices of one row for the small path (8192 ids each).
int verify_small_slices(int V) { return (V + kSliceIds - 1) / kSliceIds; }

// The batches this path takes: the plain verify (no cap-accept window) of up
// to kSmallBatchMax requests whose rows have at most kMaxBlocks sampling
// blocks.
bool verify_small_fits(int B, int V, bool audit) {
    return !audit && B <= kSmallBatchMax && (V + kSampleBlock - 1) / kSampleBlock <= kMaxBlocks;
}

cudaError_t launch_verify_small(const VerifyArgs &a, int logit_bf16, int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kSmallThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int S = verify_small_slices(a.V);
    if (logit_bf16) return cudaLaunchKernelEx(&cfg, verify_small_kernel<uint16_t>, a, S);
    return cudaLaunchKernelEx(&cfg, verify_small_kernel<float>, a, S);
}

}  // namespace dspark
