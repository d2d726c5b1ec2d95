// verify.cu -- steps a5-a6: streaming verify pass, accept / resample /
// bonus, commit.
//
// "DFlash to DSpark in SGLang", section "Background": the target checks all
// drafts in one forward, the accepted prefix is committed and the verify
// forward yields one bonus token.  "SGLang Integrates DSpark ...", section
// "The Old Problem with Speculative Decoding: It Breaks Down at Scale": the
// speculative-sampling rule (Chen et al. 2023) -- accept draft d with
// probability min(1, p(d)/q(d)); on the first rejection draw from
// norm(max(0, p - q)); "DFlash to DSpark in SGLang", section "Serving
// DeepSeek-V4 with SGLang": speculation leaves the target distribution
// unchanged.
//
// Design (GB300).  The pass is HBM-bound: every kept target row (sum L + B of
// them) and every kept draft row (sum L) is read once, V logits each.
//  * Work items are the packed target rows r (request-major, so a request's
//    rows are contiguous); item r of request b at index k < L_b is a pair
//    (target row r, draft row (b, k)); k = L_b is the bonus row.  Each item is
//    cut into 16 KB vocab tiles; a task is (item, tile).  A persistent grid
//    (2 CTAs per SM) walks the tasks round-robin, so the whole GPU sweeps the
//    requests in order.
//  * One thread per CTA issues 1-D bulk TMA copies (cp.async.bulk) of the
//    task's target tile (and draft tile) into a 3-stage shared-memory ring,
//    completing on an mbarrier with a byte count; all 256 threads consume
//    16-byte vectors from shared memory.
//  * Per tile: sampling keeps a single-pass online (max, sum) of 2^(z*s) for
//    p and q (s = log2(e)/Tm, MUFU ex2) and gathers z_p[d], z_q[d]; greedy
//    keeps (max, lowest argmax).  Warp-shuffle then block reduction; the
//    tile's record goes to the workspace.
//  * A per-request counter (atomicAdd, self-resetting) elects the CTA that
//    finishes the request's last tile; that CTA combines the records, takes
//    the accept decisions with Philox uniforms, and draws the emitted token
//    in two levels: a block of 8192 ids by its mass (u'), then an id inside
//    it (u'').  For the bonus the block masses come from the tile records,
//    so only the chosen block is read again; the residual needs one pass
//    over the rejecting row pair (streamed moments earlier, so it still sits
//    in L2) for its block masses.  Nothing ever waits on another CTA.
#include <climits>

#include "dspark_internal.cuh"

namespace dspark {
namespace {

constexpr int kVecPerChunk = kChunkBytes / 16;
static_assert(kVecPerChunk % kThreads == 0, "a tile must split evenly over the CTA");
constexpr int kStageBytes = 2 * kChunkBytes;
constexpr size_t kSmemBytes = size_t(kStages) * kStageBytes;

struct DecideSmem {
    float Mp[DSPARK_MAX_GAMMA + 1], Sp[DSPARK_MAX_GAMMA + 1];
    float Mq[DSPARK_MAX_GAMMA + 1], Sq[DSPARK_MAX_GAMMA + 1];
    int acc[DSPARK_MAX_GAMMA + 1];  // accept bits (sampling) or row argmax (greedy)
    double scan[kWarps + 1];
    float zw[2][kWarps];
    int ia, pick, pick_tid, last_tid;
    float u_blk, u_tok;
    double base;
};

struct Task {
    int r, j, b, k, Lb, pair;
    uint32_t bytes;
};

__device__ __forceinline__ Task task_of(const VerifyArgs &a, long long t) {
    Task x;
    x.r = int(t / a.nc);
    x.j = int(t - (long long)x.r * a.nc);
    x.b = a.row_req[x.r];
    x.k = a.row_k[x.r];
    x.Lb = min(max(a.L[x.b], 0), a.gamma);
    x.pair = !a.greedy && x.k < x.Lb;
    x.bytes = uint32_t(min(kChunkBytes, a.row_bytes - x.j * kChunkBytes));
    return x;
}

__device__ __forceinline__ void issue(const VerifyArgs &a, const Task &x, uint8_t *stage,
                                      uint64_t *bar) {
    const char *tsrc = static_cast<const char *>(a.target_logits) + size_t(x.r) * a.row_bytes +
                       size_t(x.j) * kChunkBytes;
    mbar_arrive_expect_tx(bar, x.bytes * (x.pair ? 2u : 1u));
    bulk_g2s(stage, tsrc, x.bytes, bar);
    if (x.pair) {
        const char *dsrc = static_cast<const char *>(a.draft_logits) +
                           (size_t(x.b) * a.gamma + x.k) * size_t(a.row_bytes) +
                           size_t(x.j) * kChunkBytes;
        bulk_g2s(stage + kChunkBytes, dsrc, x.bytes, bar);
    }
}

// Fold one vector of logits into the running (max, sum of 2^((z - max) * s)).
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

// Inclusive block scan of one double per thread; *total = block sum.
__device__ double block_incl_scan(double v, double *total, double *sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    double incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        double x = lane < kWarps ? sh[lane] : 0.0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double n = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += n;
        }
        if (lane < kWarps) sh[lane] = x;
    }
    __syncthreads();
    const double before = warp > 0 ? sh[warp - 1] : 0.0;
    *total = sh[kWarps - 1];
    __syncthreads();
    return before + incl;
}

// Sum of val(i), i < n, with the same tiling and association as find_crossing.
template <typename F>
__device__ double tiled_total(int n, F val, DecideSmem &sm) {
    double carry = 0.0;
    for (int t0 = 0; t0 < n; t0 += kThreads) {
        const int i = t0 + threadIdx.x;
        double tot;
        block_incl_scan(i < n ? double(val(i)) : 0.0, &tot, sm.scan);
        carry += tot;
    }
    return carry;
}

// Smallest i whose running sum (through i) exceeds target.  If rounding
// leaves no crossing: the last i with val(i) > 0.
template <typename F>
__device__ int find_crossing(int n, double target, F val, DecideSmem &sm) {
    const int tid = threadIdx.x;
    if (tid == 0) {
        sm.pick_tid = INT_MAX;
        sm.last_tid = -1;
    }
    __syncthreads();
    double carry = 0.0;
    for (int t0 = 0; t0 < n; t0 += kThreads) {
        const int i = t0 + tid;
        const double v = i < n ? double(val(i)) : 0.0;
        double tot;
        const double incl = carry + block_incl_scan(v, &tot, sm.scan);
        if (i < n && incl > target) atomicMin(&sm.pick_tid, i);
        if (i < n && v > 0.0) atomicMax(&sm.last_tid, i);
        carry += tot;
        __syncthreads();
        if (sm.pick_tid != INT_MAX) break;
    }
    const int idx = sm.pick_tid != INT_MAX ? sm.pick_tid : max(sm.last_tid, 0);
    __syncthreads();
    return idx;
}

// Token draw inside sampling block `blk` of a row: the smallest id whose
// running in-block weight exceeds u_tok times the block's weight.  wfn(v, w)
// fills the VE weights of 16-byte vector v of the row.  Each thread owns a
// contiguous run of vectors summed in fp32 in id order; runs are combined in
// fp64; the chosen thread re-walks its run with the same fp32 association, so
// its crossing agrees with the scan.
template <int VE, typename WF>
__device__ int block_pick(int blk, int nvec_row, float u_tok, WF wfn, DecideSmem &sm) {
    const int tid = threadIdx.x;
    const int v_begin = blk * (kSampleBlock / VE);
    const int v_end = min(nvec_row, v_begin + kSampleBlock / VE);
    const int per = (v_end - v_begin + kThreads - 1) / kThreads;
    const int t0 = min(v_end, v_begin + tid * per), t1 = min(v_end, t0 + per);
    float tsum = 0.f;
    for (int v = t0; v < t1; ++v) {
        float w[VE];
        wfn(v, w);
#pragma unroll
        for (int e = 0; e < VE; ++e) tsum += w[e];
    }
    double total;
    const double incl = block_incl_scan(double(tsum), &total, sm.scan);
    const double excl = incl - double(tsum);
    const double target = double(u_tok) * total;
    if (tid == 0) {
        sm.pick_tid = INT_MAX;
        sm.last_tid = -1;
    }
    __syncthreads();
    if (t0 < t1 && incl > target) atomicMin(&sm.pick_tid, tid);
    if (tsum > 0.f) atomicMax(&sm.last_tid, tid);
    __syncthreads();
    const int chosen = sm.pick_tid != INT_MAX ? sm.pick_tid : sm.last_tid;
    if (tid == chosen) {
        float run = 0.f;
        int pick = -1, lastpos = -1;
        for (int v = t0; v < t1 && pick < 0; ++v) {
            float w[VE];
            wfn(v, w);
#pragma unroll
            for (int e = 0; e < VE; ++e) {
                run += w[e];
                if (pick < 0 && w[e] > 0.f) {
                    lastpos = v * VE + e;
                    if (excl + double(run) > target) pick = v * VE + e;
                }
            }
        }
        sm.pick = pick >= 0 ? pick : lastpos;
    }
    if (chosen < 0 && tid == 0) sm.pick = v_begin * VE;
    __syncthreads();
    const int out = sm.pick;
    __syncthreads();
    return out;
}

__device__ void write_outputs(const VerifyArgs &a, int b, int ab, int token) {
    const int g1 = a.gamma + 1;
    for (int j = threadIdx.x; j < g1; j += kThreads) {
        int v = -1;
        if (j < ab) v = a.draft_tokens[size_t(b) * a.gamma + j];
        else if (j == ab) v = token;
        a.out_tokens[size_t(b) * g1 + j] = v;
    }
    if (threadIdx.x == 0) {
        a.accept_len[b] = ab;
        a.num_emitted[b] = ab + 1;
        if (a.seq_lens_commit) a.seq_lens_commit[b] += ab + 1;
        a.req_cnt[b] = 0;  // ready for the next launch
    }
}

// Draw from p = softmax(z / Tm) of packed target row r (global max M): the
// block masses come from the tile records of the streaming pass, so only
// the chosen block is read again.
template <typename T>
__device__ int sample_target(const VerifyArgs &a, int r, float M, float u_blk, float u_tok,
                             DecideSmem &sm) {
    constexpr int VE = Vec<T>::kElems;
    const float scale = a.scale;
    const float4 *rec = a.part + size_t(r) * a.nc;
    const int cpb = kSampleBlock / a.chunk_elems;  // tiles per sampling block
    const int nblk = (a.nc + cpb - 1) / cpb;
    auto blk_w = [&](int i) {
        float m = 0.f;
        for (int j = i * cpb; j < min(a.nc, (i + 1) * cpb); ++j) {
            const float4 x = __ldcg(rec + j);
            if (x.y > 0.f) m += x.y * exp2_approx((x.x - M) * scale);
        }
        return m;
    };
    const double total = tiled_total(nblk, blk_w, sm);
    const int blk = find_crossing(nblk, double(u_blk) * total, blk_w, sm);
    const uint4 *row = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.target_logits) +
                                                       size_t(r) * a.row_bytes);
    auto wfn = [&](int v, float (&w)[VE]) {
        float x[VE];
        Vec<T>::unpack(row[v], x);
#pragma unroll
        for (int e = 0; e < VE; ++e) w[e] = exp2_approx((x[e] - M) * scale);
    };
    return block_pick<VE>(blk, a.row_bytes / 16, u_tok, wfn, sm);
}

// Draw from norm(max(0, p - q)) at draft k of request b (packed row r); falls
// back to p when the residual mass is zero.
template <typename T>
__device__ int sample_residual(const VerifyArgs &a, int b, int k, int r, float u_blk,
                               float u_tok, DecideSmem &sm) {
    constexpr int VE = Vec<T>::kElems;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float scale = a.scale;
    const float Mp = sm.Mp[k], Mq = sm.Mq[k];
    const float iSp = 1.f / sm.Sp[k], iSq = 1.f / sm.Sq[k];
    const int nvec_row = a.row_bytes / 16;
    const uint4 *tv = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.target_logits) +
                                                      size_t(r) * a.row_bytes);
    const uint4 *dv = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.draft_logits) +
                                                      (size_t(b) * a.gamma + k) * a.row_bytes);
    auto wfn = [&](int v, float (&w)[VE]) {
        float x[VE], y[VE];
        Vec<T>::unpack(tv[v], x);
        Vec<T>::unpack(dv[v], y);
#pragma unroll
        for (int e = 0; e < VE; ++e)
            w[e] = fmaxf(0.f, exp2_approx((x[e] - Mp) * scale) * iSp -
                                  exp2_approx((y[e] - Mq) * scale) * iSq);
    };
    // Residual mass per tile, two tiles per round so 16 loads are in flight
    // per thread; the tile masses overwrite the (now unused) draft half of the
    // row's tile records.
    float *zrec = reinterpret_cast<float *>(a.part + size_t(r) * a.nc);
    constexpr int kPer = kVecPerChunk / kThreads;
    for (int c0 = 0; c0 < a.nc; c0 += 2) {
        uint4 pt[2][kPer], pd[2][kPer];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int q = 0; q < kPer; ++q) {
                const int v = (c0 + h) * kVecPerChunk + q * kThreads + tid;
                if (c0 + h < a.nc && v < nvec_row) {
                    pt[h][q] = tv[v];
                    pd[h][q] = dv[v];
                } else {
                    pt[h][q] = make_uint4(0, 0, 0, 0);
                    pd[h][q] = pt[h][q];
                }
            }
        float z[2] = {0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int q = 0; q < kPer; ++q) {
                const int v = (c0 + h) * kVecPerChunk + q * kThreads + tid;
                if (c0 + h < a.nc && v < nvec_row) {
                    float x[VE], y[VE];
                    Vec<T>::unpack(pt[h][q], x);
                    Vec<T>::unpack(pd[h][q], y);
#pragma unroll
                    for (int e = 0; e < VE; ++e)
                        z[h] += fmaxf(0.f, exp2_approx((x[e] - Mp) * scale) * iSp -
                                               exp2_approx((y[e] - Mq) * scale) * iSq);
                }
            }
        z[0] = warp_sum(z[0]);
        z[1] = warp_sum(z[1]);
        if (lane == 0) {
            sm.zw[0][warp] = z[0];
            sm.zw[1][warp] = z[1];
        }
        __syncthreads();
        if (tid < 2 && c0 + tid < a.nc) {
            double Z = 0.0;
            for (int w = 0; w < kWarps; ++w) Z += double(sm.zw[tid][w]);
            zrec[size_t(c0 + tid) * 4 + 2] = float(Z);
        }
        __syncthreads();
    }
    const int cpb = kSampleBlock / a.chunk_elems;
    const int nblk = (a.nc + cpb - 1) / cpb;
    auto blk_z = [&](int i) {
        float m = 0.f;
        for (int j = i * cpb; j < min(a.nc, (i + 1) * cpb); ++j) m += __ldcg(zrec + size_t(j) * 4 + 2);
        return m;
    };
    const double total = tiled_total(nblk, blk_z, sm);
    if (!(total > 0.0)) return sample_target<T>(a, r, Mp, u_blk, u_tok, sm);
    const int blk = find_crossing(nblk, double(u_blk) * total, blk_z, sm);
    return block_pick<VE>(blk, nvec_row, u_tok, wfn, sm);
}

template <typename T>
__device__ void decide_sampling(const VerifyArgs &a, int b, DecideSmem &sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Lb = min(max(a.L[b], 0), a.gamma), r0 = a.row_off[b], d0 = a.draft_off[b];
    const float scale = a.scale;
    for (int k = warp; k <= Lb; k += kWarps) {
        const int r = r0 + k;
        const bool pair = k < Lb;
        float mp = -INFINITY, sp = 0.f, mq = -INFINITY, sq = 0.f;
        for (int j = lane; j < a.nc; j += 32) {
            const float4 x = __ldcg(a.part + size_t(r) * a.nc + j);
            ms_combine(mp, sp, x.x, x.y, scale);
            if (pair) ms_combine(mq, sq, x.z, x.w, scale);
        }
        warp_ms_reduce(mp, sp, scale);
        if (pair) warp_ms_reduce(mq, sq, scale);
        if (lane == 0) {
            sm.Mp[k] = mp;
            sm.Sp[k] = sp;
            if (pair) {
                sm.Mq[k] = mq;
                sm.Sq[k] = sq;
                const int dt = a.draft_tokens[size_t(b) * a.gamma + k];
                float p = 0.f, q = 0.f, ratio = 0.f;
                if (dt >= 0 && dt < a.V) {
                    const float2 z = __ldcg(a.gath + r);
                    p = exp2_approx((z.x - mp) * scale) / sp;
                    q = exp2_approx((z.y - mq) * scale) / sq;
                    ratio = q > 0.f ? fminf(1.f, p / q) : 1.f;
                }
                float u, u_blk, u_tok;
                step_uniforms(a.seed, b, k, u, u_blk, u_tok);
                sm.acc[k] = u < ratio;
                a.p_tok[d0 + k] = p;
                a.q_tok[d0 + k] = q;
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        int ab = Lb;
        for (int k = 0; k < Lb; ++k)
            if (!sm.acc[k]) {
                ab = k;
                break;
            }
        float u;
        step_uniforms(a.seed, b, ab, u, sm.u_blk, sm.u_tok);
        sm.ia = ab;
    }
    __syncthreads();
    const int ab = sm.ia;
    const float u_blk = sm.u_blk, u_tok = sm.u_tok;
    const int token = ab < Lb ? sample_residual<T>(a, b, ab, r0 + ab, u_blk, u_tok, sm)
                              : sample_target<T>(a, r0 + Lb, sm.Mp[Lb], u_blk, u_tok, sm);
    write_outputs(a, b, ab, token);
}

__device__ void decide_greedy(const VerifyArgs &a, int b, DecideSmem &sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Lb = min(max(a.L[b], 0), a.gamma), r0 = a.row_off[b], d0 = a.draft_off[b];
    for (int k = warp; k <= Lb; k += kWarps) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int j = lane; j < a.nc; j += 32) {
            const float4 x = __ldcg(a.part + size_t(r0 + k) * a.nc + j);
            am_combine(bv, bi, x.x, __float_as_int(x.y));
        }
        warp_am_reduce(bv, bi);
        if (lane == 0) sm.acc[k] = bi;
    }
    for (int k = tid; k < Lb; k += kThreads) {
        a.p_tok[d0 + k] = 0.f;
        a.q_tok[d0 + k] = 0.f;
    }
    __syncthreads();
    if (tid == 0) {
        int ab = Lb;
        for (int k = 0; k < Lb; ++k)
            if (a.draft_tokens[size_t(b) * a.gamma + k] != sm.acc[k]) {
                ab = k;
                break;
            }
        sm.ia = ab;
        sm.pick = sm.acc[ab];
    }
    __syncthreads();
    write_outputs(a, b, sm.ia, sm.pick);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2) verify_kernel(const VerifyArgs a) {
    constexpr int VE = Vec<T>::kElems;
    extern __shared__ __align__(1024) uint8_t ring[];
    __shared__ uint64_t bars[kStages];
    __shared__ float red[4][kWarps];
    __shared__ int red_i[kWarps];
    __shared__ int s_last;
    __shared__ DecideSmem sm;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Packed rows as written by the compaction, never more than its capacity.
    const int n_rows = min(max(a.row_off[a.B], 0), a.B * (a.gamma + 1));
    const long long n_tasks = (long long)n_rows * a.nc;
    if ((long long)blockIdx.x >= n_tasks) return;
    const long long G = gridDim.x;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) {
        for (int i = 0; i < kStages - 1; ++i) {
            const long long t = blockIdx.x + i * G;
            if (t < n_tasks) issue(a, task_of(a, t), ring + i * kStageBytes, &bars[i]);
        }
    }

    for (int i = 0;; ++i) {
        const long long t = blockIdx.x + i * G;
        if (t >= n_tasks) break;
        const int stage = i % kStages;
        const uint32_t parity = (i / kStages) & 1;
        if (tid == 0) {
            const long long tn = t + (kStages - 1) * G;
            if (tn < n_tasks) {
                const int sn = (i + kStages - 1) % kStages;
                issue(a, task_of(a, tn), ring + sn * kStageBytes, &bars[sn]);
            }
        }
        const Task x = task_of(a, t);
        const bool ok = mbar_wait_bounded(&bars[stage], parity);
        if (!__syncthreads_and(ok)) {
            // A copy never landed: record it, drain what this CTA still has
            // in flight (bounded), and leave.
            if (tid == 0) atomicOr(a.status, kStatusWaitTimeout);
            for (int q = 0; q < kStages; ++q) {
                const long long tq = t + q * G;
                if (tq < n_tasks)
                    mbar_wait_bounded(&bars[(i + q) % kStages], ((i + q) / kStages) & 1);
            }
            return;
        }
        const uint4 *tvec = reinterpret_cast<const uint4 *>(ring + stage * kStageBytes);
        const uint4 *dvec = tvec + kVecPerChunk;
        const int nvec = int(x.bytes / 16);
        float4 rec;
        if (a.greedy) {
            float bv = -INFINITY;
            int bi = INT_MAX;
            const int y0 = x.j * a.chunk_elems;
            for (int v = tid; v < nvec; v += kThreads) {
                float z[VE];
                Vec<T>::unpack(tvec[v], z);
#pragma unroll
                for (int e = 0; e < VE; ++e)
                    if (z[e] > bv) {
                        bv = z[e];
                        bi = y0 + v * VE + e;
                    }
            }
            warp_am_reduce(bv, bi);
            if (lane == 0) {
                red[0][warp] = bv;
                red_i[warp] = bi;
            }
            __syncthreads();
            if (warp == 0) {
                bv = lane < kWarps ? red[0][lane] : -INFINITY;
                bi = lane < kWarps ? red_i[lane] : INT_MAX;
                warp_am_reduce(bv, bi);
            }
            rec = make_float4(bv, __int_as_float(bi), 0.f, 0.f);
        } else {
            const float scale = a.scale;
            float mp = -INFINITY, sp = 0.f, mq = -INFINITY, sq = 0.f;
            if (x.pair) {
                for (int v = tid; v < nvec; v += kThreads) {
                    float z[VE];
                    Vec<T>::unpack(tvec[v], z);
                    online_update<VE>(mp, sp, z, scale);
                    Vec<T>::unpack(dvec[v], z);
                    online_update<VE>(mq, sq, z, scale);
                }
            } else {
                for (int v = tid; v < nvec; v += kThreads) {
                    float z[VE];
                    Vec<T>::unpack(tvec[v], z);
                    online_update<VE>(mp, sp, z, scale);
                }
            }
            warp_ms_reduce(mp, sp, scale);
            if (x.pair) warp_ms_reduce(mq, sq, scale);
            if (lane == 0) {
                red[0][warp] = mp;
                red[1][warp] = sp;
                red[2][warp] = mq;
                red[3][warp] = sq;
            }
            __syncthreads();
            if (warp == 0) {
                mp = lane < kWarps ? red[0][lane] : -INFINITY;
                sp = lane < kWarps ? red[1][lane] : 0.f;
                mq = lane < kWarps ? red[2][lane] : -INFINITY;
                sq = lane < kWarps ? red[3][lane] : 0.f;
                warp_ms_reduce(mp, sp, scale);
                warp_ms_reduce(mq, sq, scale);
            }
            rec = make_float4(mp, sp, mq, sq);
            if (tid == 0 && x.pair) {
                const int dt = a.draft_tokens[size_t(x.b) * a.gamma + x.k];
                const int y0 = x.j * a.chunk_elems;
                if (dt >= y0 && dt < y0 + nvec * VE) {
                    const float zp = Vec<T>::load1(tvec, dt - y0);
                    const float zq = Vec<T>::load1(dvec, dt - y0);
                    a.gath[x.r] = make_float2(zp, zq);
                }
            }
        }
        if (tid == 0) {
            a.part[size_t(x.r) * a.nc + x.j] = rec;
            __threadfence();
            const int total = (x.Lb + 1) * a.nc;
            s_last = atomicAdd(&a.req_cnt[x.b], 1) == total - 1;
        }
        __syncthreads();  // the stage is free again; s_last is visible
        if (s_last) {
            __threadfence();
            if (a.greedy) decide_greedy(a, x.b, sm);
            else decide_sampling<T>(a, x.b, sm);
            __syncthreads();
        }
    }
}

template <typename T>
cudaError_t set_smem_attr() {
    return cudaFuncSetAttribute(verify_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(kSmemBytes));
}

}  // namespace

size_t verify_smem_bytes() { return kSmemBytes; }

int verify_blocks_per_sm(int logit_bf16) {
    cudaError_t e = logit_bf16 ? set_smem_attr<uint16_t>() : set_smem_attr<float>();
    if (e != cudaSuccess) return -1;
    int n = 0;
    e = logit_bf16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, verify_kernel<uint16_t>,
                                                                   kThreads, kSmemBytes)
                   : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, verify_kernel<float>,
                                                                   kThreads, kSmemBytes);
    return e == cudaSuccess ? n : -1;
}

cudaError_t launch_verify(const VerifyArgs &a, int logit_bf16, int grid, cudaStream_t s) {
    if (logit_bf16)
        verify_kernel<uint16_t><<<grid, kThreads, kSmemBytes, s>>>(a);
    else
        verify_kernel<float><<<grid, kThreads, kSmemBytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace dspark
