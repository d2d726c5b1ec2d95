// score_budget.cu -- steps a1-a3 and the scans of a4 in one kernel (and,
// for dspark_score_compact, the packing of a4 as well).
//
// "DFlash to DSpark in SGLang", section "DSpark: a sequential head and a
// verify budget": a linear projection plus sigmoid on the drafter hidden
// state scores each draft; the product across the block is the survival
// probability; Sequential Temperature Scaling calibrates it.  Section "The
// confidence scheduler and verify modes": walk down the survival curve and
// stop where the gain no longer covers the marginal cost c.  Section
// "Zero-overhead scheduling and kernels": a verify-length top-k schedule
// bounds the batch.
//
// Work split.  One CTA per resident slot.  A producer warp claims hidden rows
// one at a time from a device counter and streams them through a ring of
// 16 KB shared-memory stages with 1-D bulk TMA copies; eight consumer warps
// take the stages in the same order, 16-byte vectors interleaved over their
// 256 threads, and accumulate fp32 dot products against the head weight.
// When a row fits one stage every row puts the same vectors of d on a thread,
// so the thread keeps its slice of the weight in registers; longer rows read
// it through L1.  At a row's last tile the last warp to finish sums the eight
// warp partials in a fixed order and writes the row's confidence (bias,
// 1/tau_i, sigmoid).  The CTA that publishes the batch's last rows (row
// counter) then forms, one thread per request, the cumulative product S and
// the pre-cap length L0_b, and runs the cap: an
// MSB-first radix select over the fp32 bit patterns of the candidate gains
// S_{b,k} (non-negative floats order like their bit patterns), ties resolved
// by request then position, followed by the exclusive scans and, when asked,
// the ragged packing.  Up to 256 requests this finish keeps everything on
// chip (finish_fast); larger batches take finish_general.  Counters reset
// themselves, so no CTA waits on another and the kernel is safe to replay.
//
// score_entropy_kernel is the same kernel with the draft logit rows as its
// rows and an entropy consumer in place of the dot product: the confidence of
// a draft is exp(-H) of its distribution ("SGLang Integrates DSpark ...",
// "DSpark's Core Idea: Only Verify the Parts You're Confident About").
#include <algorithm>

#include "dspark_internal.cuh"

namespace dspark {
namespace {

// Barrier of the 256 threads (warps 0-7) that run the scans and the cap; in
// the streaming kernel the producer warp does not take part.
__device__ __forceinline__ void sync256() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Block-wide exclusive scan of one int per thread; *total gets the sum.
// `sh` needs kWarps + 1 ints.  Called by warps 0-7 together (sync256).
__device__ int block_excl_scan_int(int v, int *total, int *sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) sh[warp] = incl;
    sync256();
    if (warp == 0) {
        int x = lane < kWarps ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += n;
        }
        if (lane < kWarps) sh[lane] = x;
    }
    sync256();
    const int before = warp > 0 ? sh[warp - 1] : 0;
    *total = sh[kWarps - 1];
    sync256();
    return before + incl - v;
}

// Exclusive scans of L into draft_off and row_off (row_off = draft_off + b).
__device__ void write_offsets(int B, const int32_t *L, int32_t *draft_off, int32_t *row_off,
                              int *sh) {
    int carry = 0;
    for (int base = 0; base < B; base += kThreads) {
        const int b = base + threadIdx.x;
        const int v = b < B ? L[b] : 0;
        int total;
        const int ex = block_excl_scan_int(v, &total, sh);
        if (b < B) {
            draft_off[b] = carry + ex;
            row_off[b] = carry + ex + b;
        }
        carry += total;
    }
    if (threadIdx.x == 0) {
        draft_off[B] = carry;
        row_off[B] = carry + B;
    }
}

// A hint to bring the 128-byte line holding p into L2.
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

constexpr int kScoreStages = 4;
constexpr int kScoreTile = 16384;                   // bytes per stage
constexpr int kScoreThreads = (kWarps + 1) * 32;    // 8 consumer warps + producer
constexpr int kScoreVecPerThread = kScoreTile / 16 / kThreads;
constexpr size_t kScoreSmemBytes = size_t(kScoreStages) * kScoreTile;

struct ScoreSmem {
    uint64_t full[kScoreStages], empty[kScoreStages];
    int row[kScoreStages];             // hidden row of the stage (-1: no more rows)
    int tile[kScoreStages];            // its tile within the row
    float part[kScoreStages][kWarps];  // warp partials of a row's last tile
    int done[kScoreStages];            // warps past a row's last tile
    int run_cap;                       // this CTA finished the batch
};

struct RowShape {
    int rows;       // B * gamma
    int ntr;        // tiles per row
    int row_bytes;
};

__device__ __forceinline__ RowShape row_shape(const ScoreArgs &a, int elem_bytes) {
    RowShape rs;
    rs.rows = a.B * a.gamma;
    rs.row_bytes = a.d * elem_bytes;
    rs.ntr = (rs.row_bytes + kScoreTile - 1) / kScoreTile;
    return rs;
}

// Lane 0 of warp 8.  Starts on row blockIdx.x, then claims rows one at a
// time from a device counter (the next claim is in flight while the current
// row is copied), so every CTA streams until the batch runs out.
__device__ void score_producer(const ScoreArgs &a, ScoreSmem &sm, uint8_t *ring,
                               const RowShape &rs) {
    const char *hidden = static_cast<const char *>(a.hidden);
    int next = blockIdx.x;  // the first row needs no claim
    for (int fill = 0;;) {
        const int r = next;
        // (a grid with a CTA per row has nothing to claim: no round trip)
        if (r < rs.rows)
            next = rs.rows <= int(gridDim.x) ? rs.rows : int(gridDim.x) + atomicAdd(a.row_ctr, 1);
        for (int q = 0; q < (r < rs.rows ? rs.ntr : 1); ++q, ++fill) {
            const int s = fill % kScoreStages, n = fill / kScoreStages;
            if (n > 0 && !mbar_wait_bounded(&sm.empty[s], (n - 1) & 1, a.wait_ns)) {
                atomicOr(a.status, kStatusWaitTimeout);
                // Leave only once every copy issued into the ring has landed.
                for (int f = max(0, fill - kScoreStages); f < fill; ++f)
                    mbar_wait_bounded(&sm.full[f % kScoreStages], (f / kScoreStages) & 1,
                                      kDrainTimeoutNs);
                return;
            }
            if (r >= rs.rows) {
                sm.row[s] = -1;
                mbar_arrive(&sm.full[s]);
                return;
            }
            sm.row[s] = r;
            sm.tile[s] = q;
            const int bytes = min(kScoreTile, rs.row_bytes - q * kScoreTile);
            mbar_arrive_expect_tx(&sm.full[s], uint32_t(bytes));
            bulk_g2s(ring + size_t(s) * kScoreTile,
                     hidden + size_t(r) * rs.row_bytes + size_t(q) * kScoreTile, uint32_t(bytes),
                     &sm.full[s]);
        }
    }
}

// Warps 0-7.  Returns the number of rows this CTA published.
template <typename T>
__device__ int score_consumer(const ScoreArgs &a, ScoreSmem &sm, const uint8_t *ring,
                              const RowShape &rs, int warp, int lane) {
    constexpr int VE = Vec<T>::kElems;
    constexpr int NV = kScoreVecPerThread;
    constexpr int kTileElems = kScoreTile / int(sizeof(T));
    const int tid = warp * 32 + lane;
    // A row that fits one tile puts the same vectors of d on this thread in
    // every row: its slice of the head weight then stays in registers.
    const bool w_regs = rs.ntr == 1;
    float wr[NV][VE];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int v = tid + kThreads * i;
#pragma unroll
        for (int j = 0; j < VE; j += 4) {
            float4 wv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (w_regs && v * VE < a.d)
                wv = __ldg(reinterpret_cast<const float4 *>(a.head_w) + (v * VE + j) / 4);
            wr[i][j] = wv.x;
            wr[i][j + 1] = wv.y;
            wr[i][j + 2] = wv.z;
            wr[i][j + 3] = wv.w;
        }
    }
    int nrows = 0;
    float acc = 0.f;
    for (int fill = 0;; ++fill) {
        const int s = fill % kScoreStages, n = fill / kScoreStages;
        if (!mbar_wait_bounded(&sm.full[s], n & 1, a.wait_ns)) {
            if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
            return nrows;
        }
        const int r = sm.row[s], q = sm.tile[s];
        if (r < 0) return nrows;
        if (q == 0) acc = 0.f;
        // The row's bias and temperature are needed at its end; load them
        // now, behind the FMAs.
        const int rb = r / a.gamma;
        const bool last_tile = q + 1 == rs.ntr;
        const float bias = last_tile ? __ldg(&a.head_bias[rb]) : 0.f;
        const float tau = last_tile ? __ldg(&a.sts_tau[r - rb * a.gamma]) : 1.f;
        const int nvec = min(kScoreTile, rs.row_bytes - q * kScoreTile) / 16;
        const uint4 *tv = reinterpret_cast<const uint4 *>(ring + size_t(s) * kScoreTile);
        uint4 x[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int v = tid + kThreads * i;
            x[i] = v < nvec ? tv[v] : make_uint4(0, 0, 0, 0);
        }
        if (w_regs) {
            // Vectors past the row are zero in both x and wr.
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                float e[VE];
                Vec<T>::unpack(x[i], e);
#pragma unroll
                for (int j = 0; j < VE; ++j) acc = fmaf(e[j], wr[i][j], acc);
            }
        } else {
            const float4 *w4 = reinterpret_cast<const float4 *>(a.head_w + size_t(q) * kTileElems);
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int v = tid + kThreads * i;
                if (v < nvec) {
                    float e[VE];
                    Vec<T>::unpack(x[i], e);
#pragma unroll
                    for (int j = 0; j < VE; j += 4) {
                        const float4 wv = __ldg(w4 + (v * VE + j) / 4);
                        acc = fmaf(e[j], wv.x, acc);
                        acc = fmaf(e[j + 1], wv.y, acc);
                        acc = fmaf(e[j + 2], wv.z, acc);
                        acc = fmaf(e[j + 3], wv.w, acc);
                    }
                }
            }
        }
        if (q + 1 < rs.ntr) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
            continue;
        }
        // Last tile of row r: the last warp here sums the eight partials.
        ++nrows;
        const float wsum = warp_sum(acc);
        int last = 0;
        if (lane == 0) {
            sm.part[s][warp] = wsum;
            __threadfence_block();
            last = atomicAdd(&sm.done[s], 1) == kWarps - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
            continue;
        }
        __threadfence_block();
        float dot = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) dot += sm.part[s][w];
        __syncwarp();
        if (lane == 0) {
            sm.done[s] = 0;
            mbar_arrive(&sm.empty[s]);
            // conf = sigmoid((w . h + bias_b) / tau_i) of this row
            const float x = (dot + bias) / tau;
            a.conf[r] = 1.f / (1.f + expf(-x));
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// Entropy-confidence variant ("SGLang Integrates DSpark ...", "DSpark's Core
// Idea: Only Verify the Parts You're Confident About": a low-entropy draft
// distribution is a confident one).  conf = exp(-H(q)), q = softmax(z / theta),
// over the draft logit row of each draft.  The rows stream through the same
// ring; each thread keeps, in log2 units y = z log2(e) / theta,
//   m = max y,  s = sum 2^(y - m),  t = sum 2^(y - m) (y - m),
// so that H = ln 2 (log2 s - t / s) and conf = 2^(t / s) / s.
// ---------------------------------------------------------------------------
struct Ent {
    float m, s, t;
};

// Bring both onto the larger maximum and add.  An empty side (s = 0, no
// finite logit seen, m = -inf) is skipped.
__device__ __forceinline__ Ent ent_join(Ent a, Ent b) {
    if (!(a.s > 0.f)) return b;
    if (!(b.s > 0.f)) return a;
    const float M = fmaxf(a.m, b.m);
    const float da = a.m - M, db = b.m - M;
    const float fa = exp2_approx(da), fb = exp2_approx(db);
    Ent r;
    r.m = M;
    r.s = a.s * fa + b.s * fb;
    r.t = fa * fmaf(da, a.s, a.t) + fb * fmaf(db, b.s, b.t);
    return r;
}

__device__ __forceinline__ Ent ent_warp_reduce(Ent e) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Ent x;
        x.m = __shfl_xor_sync(0xffffffffu, e.m, o);
        x.s = __shfl_xor_sync(0xffffffffu, e.s, o);
        x.t = __shfl_xor_sync(0xffffffffu, e.t, o);
        e = ent_join(e, x);
    }
    return e;
}

// Warps 0-7 of the entropy kernel.  Returns the number of rows published.
template <typename T>
__device__ int entropy_consumer(const ScoreArgs &a, ScoreSmem &sm, const uint8_t *ring,
                                const RowShape &rs, int warp, int lane) {
    constexpr int VE = Vec<T>::kElems;
    constexpr int NV = kScoreVecPerThread;
    __shared__ float4 part[kScoreStages][kWarps];
    const int tid = warp * 32 + lane;
    const float scale = a.ent_scale;
    int nrows = 0;
    Ent acc{-INFINITY, 0.f, 0.f};
    for (int fill = 0;; ++fill) {
        const int s = fill % kScoreStages, n = fill / kScoreStages;
        if (!mbar_wait_bounded(&sm.full[s], n & 1, a.wait_ns)) {
            if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
            return nrows;
        }
        const int r = sm.row[s], q = sm.tile[s];
        if (r < 0) return nrows;
        if (q == 0) acc = Ent{-INFINITY, 0.f, 0.f};
        const int nvec = min(kScoreTile, rs.row_bytes - q * kScoreTile) / 16;
        const uint4 *tv = reinterpret_cast<const uint4 *>(ring + size_t(s) * kScoreTile);
        uint4 x[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int v = tid + kThreads * i;
            x[i] = v < nvec ? tv[v] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            if (tid + kThreads * i >= nvec) continue;
            float z[VE];
            Vec<T>::unpack(x[i], z);
            float zv = z[0];
#pragma unroll
            for (int j = 1; j < VE; ++j) zv = fmaxf(zv, z[j]);
            const float mv = zv * scale;
            if (mv > acc.m) {
                if (acc.s > 0.f) {  // acc.m is finite once anything was added
                    const float dm = acc.m - mv;
                    const float f = exp2_approx(dm);
                    acc.t = f * fmaf(dm, acc.s, acc.t);
                    acc.s *= f;
                }
                acc.m = mv;
            }
            // dy = y - m, floored at -200: 2^dy is then 0 in fp32 (as it is for
            // any dy below -150), so -inf logits (masked ids), and -inf - -inf
            // while nothing finite has been seen (fmaxf drops the NaN), add
            // nothing.  Per vector, the weights are summed pairwise and the
            // weighted offsets in one fused chain, then both join the running
            // sums (short rounding chains, one FFMA per term for t).
            float p[VE], tv = 0.f;
#pragma unroll
            for (int j = 0; j < VE; ++j) {
                const float dy = fmaxf(fmaf(z[j], scale, -acc.m), -200.f);
                p[j] = exp2_approx(dy);
                tv = fmaf(p[j], dy, tv);
            }
#pragma unroll
            for (int st = 1; st < VE; st <<= 1)
#pragma unroll
                for (int j = 0; j + st < VE; j += 2 * st) p[j] += p[j + st];
            acc.s += p[0];
            acc.t += tv;
        }
        if (q + 1 < rs.ntr) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
            continue;
        }
        // Last tile of row r: the last warp here joins the eight partials.
        ++nrows;
        const Ent w = ent_warp_reduce(acc);
        int last = 0;
        if (lane == 0) {
            part[s][warp] = make_float4(w.m, w.s, w.t, 0.f);
            __threadfence_block();
            last = atomicAdd(&sm.done[s], 1) == kWarps - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
            continue;
        }
        __threadfence_block();
        Ent tot{-INFINITY, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < kWarps; ++k) {
            const float4 pk = part[s][k];
            tot = ent_join(tot, Ent{pk.x, pk.y, pk.z});
        }
        __syncwarp();
        if (lane == 0) {
            sm.done[s] = 0;
            mbar_arrive(&sm.empty[s]);
            // conf = exp(-H) = 2^(t / s) / s, at most 1 (a one-hot row's
            // rounding may leave t a hair above 0)
            a.conf[r] = fminf(1.f, exp2f(tot.t / tot.s) / tot.s);
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// Request curves and the cap, run by the CTA that publishes the batch's last
// row (warps 0-7).  Its 64 KB ring is free by then.  When B * pitch <=
// kOnChip (pitch = gamma rounded up to odd, so a thread per request reads
// its row without bank conflicts) it holds
//   [0, 32 KB)   confidences, [b * pitch + k];
//   [32, 64 KB)  S_{b,k+1}, same layout;
// and once the confidences are written out, the radix select's two lists of
// kListCap keys take [0, 32 KB).  Larger batches work from global memory.
// ---------------------------------------------------------------------------
constexpr int kListCap = 4096;
constexpr int kOnChip = 8192;
static_assert(2 * kListCap * 4 <= kOnChip * 4 && 2 * kOnChip * 4 <= int(kScoreSmemBytes),
              "the finishing CTA's ring layout");

struct FinishSmem {
    int sh[kWarps + 1];
    unsigned hist[256];
    int sel[2];
    int cnt;
};

// Thread-per-request survival curve: S_0 = 1, S_k = S_{k-1} * conf_k, and
// L0_b = max{k : S_k >= c} (0 if none).  With sC/sS the confidences come
// from and the curve goes to shared memory (the caller writes it out);
// otherwise global memory is used directly.
__device__ int request_curve(const ScoreArgs &a, int b, const float *sC, float *sS, int pitch) {
    const int g = a.gamma;
    float S = 1.f;
    int L = 1.f >= a.cost_c ? 0 : -1;
    for (int k0 = 0; k0 < g; k0 += 8) {
        float cv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int k = k0 + j;
            cv[j] = k >= g ? 0.f : sC ? sC[b * pitch + k] : __ldcg(&a.conf[size_t(b) * g + k]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int k = k0 + j;
            if (k < g) {
                S *= cv[j];
                if (sS) sS[b * pitch + k] = S;
                else a.survival[size_t(b) * g + k] = S;
                if (S >= a.cost_c) L = k + 1;
            }
        }
    }
    const int l0 = L < 0 ? 0 : L;
    a.L0[b] = l0;
    return l0;
}

// L0_b recounted from the shared curve: S does not increase with k (each
// factor is at most 1 and rounding is monotone), so the k with S_k >= c are
// exactly 1..L0_b.
__device__ __forceinline__ int l0_of(const ScoreArgs &a, const float *sS, int pitch, int b) {
    if (!sS) return __ldcg(&a.L0[b]);
    int n = 0;
    for (int k = 0; k < a.gamma; ++k) n += sS[b * pitch + k] >= a.cost_c;
    return n;
}

// Bit pattern of S_{b,k+1}, from the shared copy when there is one.
__device__ __forceinline__ unsigned s_key(const ScoreArgs &a, const float *sS, int pitch, int b,
                                          int k) {
    return __float_as_uint(sS ? sS[b * pitch + k] : __ldcg(&a.survival[size_t(b) * a.gamma + k]));
}

// Warp-aggregated histogram add: the lanes of the first two bins present
// add once per bin (keys cluster in a few bins in the first passes), the
// rest one by one (then they are spread over many bins).
__device__ __forceinline__ void hist_add(unsigned *hist, bool hit, unsigned bin, int lane) {
    unsigned rem = __ballot_sync(0xffffffffu, hit);
#pragma unroll
    for (int round = 0; round < 2; ++round) {
        if (rem == 0u) return;
        const int lead = __ffs(rem) - 1;
        const unsigned lb = __shfl_sync(0xffffffffu, bin, lead);
        const unsigned same = __ballot_sync(0xffffffffu, hit && bin == lb);
        if (lane == lead) atomicAdd(&hist[lb], unsigned(__popc(same)));
        rem &= ~same;
    }
    if (rem & (1u << lane)) atomicAdd(&hist[bin], 1u);
}

// Warp 0 finds the digit holding the need-th largest key; fs.sel gets the
// digit and the rank still to place within it.
__device__ void select_digit(FinishSmem &fs, int need, int tid) {
    if (tid >= 32) return;
    // lane l owns bins 8l .. 8l+7; suffix sums from the top bin down
    unsigned local = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) local += fs.hist[tid * 8 + q];
    unsigned suf = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned n = __shfl_down_sync(0xffffffffu, suf, o);
        if (tid + o < 32) suf += n;
    }
    const unsigned above = suf - local;  // keys in bins above this lane's
    if (above < unsigned(need) && unsigned(need) <= suf) {
        unsigned cum = above;
        for (int q = 7; q >= 0; --q) {
            const unsigned c = fs.hist[tid * 8 + q];
            if (cum + c >= unsigned(need)) {
                fs.sel[0] = tid * 8 + q;
                fs.sel[1] = need - int(cum);
                break;
            }
            cum += c;
        }
    }
}

// Step a4 in the finishing CTA of the general path, slot by slot as the
// compaction kernel does it: slot (b, j) of the B*(gamma+1) capacity writes
// packed row row_off[b] + j when j <= L_b, and slot t >= N_rows writes the
// padding of row t.  L and row_off were written by this CTA.
__device__ void pack_slots(const ScoreArgs &a) {
    const int g1 = a.gamma + 1, cap = a.B * g1;
    const int n_rows = a.row_off[a.B];
    for (int t = threadIdx.x; t < cap; t += kThreads) {
        const int b = t / g1, j = t - b * g1;
        if (j <= a.L[b]) {
            const int r = a.row_off[b] + j;
            a.packed_ids[r] = j == 0 ? (a.last_tokens ? a.last_tokens[b] : -1)
                                     : a.draft_tokens[size_t(b) * a.gamma + j - 1];
            a.packed_pos[r] = (a.seq_lens ? a.seq_lens[b] : 0) + j;
            a.row_req[r] = b;
            a.row_k[r] = j;
        }
        if (t >= n_rows) {
            a.packed_ids[t] = -1;
            a.packed_pos[t] = 0;
            a.row_req[t] = -1;
            a.row_k[t] = -1;
        }
    }
}

__device__ void finish_general(const ScoreArgs &a, uint8_t *ring) {
    __shared__ FinishSmem fs;
    const int B = a.B, g = a.gamma, tid = threadIdx.x, lane = tid & 31;
    const int pitch = g | 1;
    const bool on_chip = (long long)B * pitch <= kOnChip;
    float *sC = on_chip ? reinterpret_cast<float *>(ring) : nullptr;
    float *sS = on_chip ? reinterpret_cast<float *>(ring) + kOnChip : nullptr;
    unsigned *listA = reinterpret_cast<unsigned *>(ring);
    unsigned *listB = listA + kListCap;
    const int n_rows = B * g;
    if (on_chip) {
        // Coalesced read of every confidence into the per-request layout.
        for (int base = 0; base < n_rows; base += 16 * kThreads) {
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = base + j * kThreads + tid;
                v[j] = i < n_rows ? __ldcg(&a.conf[i]) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = base + j * kThreads + tid;
                if (i < n_rows) {
                    const int b = i / g;
                    sC[b * pitch + (i - b * g)] = v[j];
                }
            }
        }
    }
    sync256();
    for (int b = tid; b < B; b += kThreads) request_curve(a, b, sC, sS, pitch);
    sync256();
    if (on_chip) {
        // Coalesced write of the survival curves.
        for (int i = tid; i < n_rows; i += kThreads) {
            const int b = i / g;
            a.survival[i] = sS[b * pitch + (i - b * g)];
        }
    }

    // Each request's candidate keys S_{b,1..L0_b} go to listA at the
    // exclusive scan of L0 (while they fit); listA overwrites the staged
    // confidences, which the barrier inside the scan retires.
    int sum = 0;
    for (int base = 0; base < B; base += kThreads) {
        const int b = base + tid;
        const int l0 = b < B ? l0_of(a, sS, pitch, b) : 0;
        int total;
        const int off = sum + block_excl_scan_int(l0, &total, fs.sh);
        for (int k = 0; k < l0 && off + k < kListCap; ++k) listA[off + k] = s_key(a, sS, pitch, b, k);
        sum += total;
    }
    sync256();

    if (a.cap_T < 0 || sum <= a.cap_T) {
        for (int b = tid; b < B; b += kThreads) a.L[b] = l0_of(a, sS, pitch, b);
    } else if (a.cap_T == 0) {
        for (int b = tid; b < B; b += kThreads) a.L[b] = 0;
    } else {
        // The cap_T-th largest key, 8 bits per pass from the top.
        unsigned prefix = 0, mask = 0;
        int need = a.cap_T;  // rank still to place within keys matching `prefix`
        const bool listed = sum <= kListCap;
        unsigned *src = listA, *dst = listB;
        int n = sum;
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            for (int i = tid; i < 256; i += kThreads) fs.hist[i] = 0;
            if (tid == 0) {
                fs.sel[0] = 0;
                fs.sel[1] = need;
                fs.cnt = 0;
            }
            sync256();
            if (listed) {
                // The list holds exactly the keys that match `prefix`.
                for (int base = 0; base < n; base += kThreads) {
                    const int i = base + tid;
                    const unsigned kv = i < n ? src[i] : 0u;
                    hist_add(fs.hist, i < n, (kv >> shift) & 255u, lane);
                }
            } else {
                for (int base = 0; base < B; base += kThreads) {
                    const int b = base + tid;
                    const int l0 = b < B ? l0_of(a, sS, pitch, b) : 0;
                    for (int k = 0; k < g; ++k) {
                        const unsigned kv = k < l0 ? s_key(a, sS, pitch, b, k) : 0u;
                        hist_add(fs.hist, k < l0 && (kv & mask) == prefix, (kv >> shift) & 255u, lane);
                    }
                }
            }
            sync256();
            select_digit(fs, need, tid);
            sync256();
            const unsigned d = unsigned(fs.sel[0]);
            need = fs.sel[1];
            prefix |= d << shift;
            mask |= 255u << shift;
            if (listed && pass < 3) {
                // Keep the keys of the chosen digit for the next pass.
                for (int base = 0; base < n; base += kThreads) {
                    const int i = base + tid;
                    const unsigned kv = i < n ? src[i] : 0u;
                    const bool keep = i < n && ((kv >> shift) & 255u) == d;
                    const unsigned bal = __ballot_sync(0xffffffffu, keep);
                    if (bal) {
                        const int lead = __ffs(bal) - 1;
                        int pos = 0;
                        if (lane == lead) pos = atomicAdd(&fs.cnt, __popc(bal));
                        pos = __shfl_sync(0xffffffffu, pos, lead);
                        if (keep) dst[pos + __popc(bal & ((1u << lane) - 1u))] = kv;
                    }
                }
                sync256();
                n = fs.cnt;
                unsigned *t = src;
                src = dst;
                dst = t;
            }
            sync256();
        }
        // prefix is the threshold key; `need` keys equal to it are kept, the
        // lowest (b, k) first.  Within a request keys do not increase with k,
        // so the kept set of each request is a prefix.
        int carry = 0;
        for (int base = 0; base < B; base += kThreads) {
            const int b = base + tid;
            int above = 0, equal = 0;
            if (b < B) {
                const int l0 = l0_of(a, sS, pitch, b);
                for (int k = 0; k < l0; ++k) {
                    const unsigned key = s_key(a, sS, pitch, b, k);
                    above += key > prefix;
                    equal += key == prefix;
                }
            }
            int total;
            const int ex = block_excl_scan_int(equal, &total, fs.sh);
            if (b < B) {
                const int keep = min(max(need - (carry + ex), 0), equal);
                a.L[b] = above + keep;
            }
            carry += total;
        }
    }
    sync256();
    write_offsets(B, a.L, a.draft_off, a.row_off, fs.sh);
    if (a.pack) {
        sync256();  // L and row_off, written above by this CTA, are read back
        pack_slots(a);
    }
}

// ---------------------------------------------------------------------------
// Fast finish: B <= kThreads, one request per thread, everything in the
// ring.  The same outputs as finish_general, with fewer round trips:
//   * each thread loads its request's gamma confidences straight into
//     registers, forms S_{b,1..gamma} and L0_b there and keeps the keys
//     S_{b,1..L0_b} in shared memory at b * pitch;
//   * one block reduction gives sum L0, the largest key (some S_{b,1}) and
//     the smallest (some S_{b,L0_b});
//   * the cap's radix select (fast_select) takes 4-bit digits from the
//     first bit in which those two differ, counted in registers, one
//     barrier a pass, until at most 32 candidates are left, which every
//     warp then finishes bit by bit with ballots.  (Measured on the B = 256
//     shape: 8-bit digits counted by shared atomics serialised on the few
//     bins the clustered keys fall into, ~1.4 us a pass; 4-bit passes to
//     the last bit cost ~0.4-0.7 us each, seven of them.)
//   * the packing (when asked for) reads the draft tokens, last tokens and
//     cached lengths into shared memory at the start, behind the
//     confidences, and writes the packed rows coalesced at the end.
// Ring layout in 32-bit words:
//   [0, B * pitch)                     keys S_{b,k+1} at b * pitch + k
//   [tok, + B * gamma)                 draft tokens      } packing only
//   [last, + B), [seq, + B)            last tokens, cached lengths
// and, after the cap, [0, cap) the request of each packed row and
// [cap, cap + B) the row offsets (cap = B * (gamma + 1)).
// ---------------------------------------------------------------------------
constexpr int kRingWords = int(kScoreSmemBytes / 4);

struct FastLayout {
    int tok, last, seq, roff, total;
};

__device__ __forceinline__ FastLayout fast_layout(int B, int g, int pack) {
    FastLayout f;
    const int pitch = g | 1, cap = B * (g + 1);
    f.roff = cap;
    f.tok = pack ? max(B * pitch, cap + B) : B * pitch;
    f.last = f.tok + (pack ? B * g : 0);
    f.seq = f.last + (pack ? B : 0);
    f.total = f.seq + (pack ? B : 0);
    return f;
}

__device__ __forceinline__ bool fast_finish_fits(const ScoreArgs &a) {
    return a.B <= kThreads && fast_layout(a.B, a.gamma, a.pack).total <= kRingWords;
}

struct FastSmem {
    int red[kWarps][3];         // per-warp sum of L0, largest key, smallest key
    unsigned wh[2][kWarps][8];  // per-warp digit counts, two 16-bit bins a word,
                                // by pass parity
    unsigned cand[32];          // the last <= 32 candidate keys of the select
    int ncand;                  // their count, as they are gathered
    int sh[kWarps + 1];         // block scans
};

// Copy n ints from global to shared, 16 loads in flight per thread.
__device__ __forceinline__ void stage_ints(int *dst, const int32_t *src, int n) {
    for (int base = 0; base < n; base += 16 * kThreads) {
        int v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int i = base + j * kThreads + int(threadIdx.x);
            v[j] = i < n ? __ldg(src + i) : 0;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int i = base + j * kThreads + int(threadIdx.x);
            if (i < n) dst[i] = v[j];
        }
    }
}

// Confidences k0 .. k0 + 15 of one request (0 past gamma): four 16-byte
// loads when gamma % 4 == 0 and the rows are 16-byte aligned.
__device__ __forceinline__ void load_conf16(const float *crow, int k0, int g, bool vec,
                                            float (&c)[16]) {
    if (vec) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k0 + 4 * q < g) v = __ldcg(reinterpret_cast<const float4 *>(crow + k0) + q);
            c[4 * q] = v.x;
            c[4 * q + 1] = v.y;
            c[4 * q + 2] = v.z;
            c[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) c[j] = k0 + j < g ? __ldcg(crow + k0 + j) : 0.f;
    }
}

// Add a key's 4-bit digit at `shift` to a thread's 16 byte-wide bins (h0:
// digits 0-7, h1: 8-15; a request has at most 64 keys, so no byte
// overflows) when the key is valid and matches the prefix.
__device__ __forceinline__ void count_digit(unsigned key, bool valid, unsigned mask,
                                            unsigned prefix, int shift,
                                            unsigned long long &h0, unsigned long long &h1) {
    if (valid && (key & mask) == prefix) {
        const unsigned dg = (key >> shift) & 15u;
        const unsigned long long inc = 1ull << ((dg & 7u) * 8u);
        if (dg & 8u) h1 += inc;
        else h0 += inc;
    }
}

// The cap_T-th largest key (as bits) and how many keys equal to it are
// kept, over the keys of every request (thread b: S_{b,1..l0}, in the
// registers c[] when gamma <= 16, else srow[0, l0)).
//
// Four bits a pass, from the first bit in which the largest and smallest key
// differ (every key shares the bits above).  A request's keys do not
// increase with k, so the keys that match a prefix form one run
// [lo_b, hi_b) of its list and a thread counts only that run, into byte
// bins in registers.  The warps sum the bins (16-bit fields, one reduction
// per two bins) and write them to shared memory; after one barrier every
// warp reads all eight and picks the digit itself by a suffix scan, so one
// barrier a pass suffices (the counts are double-buffered by pass).  Once
// the chosen digit holds at most 32 keys, those keys are gathered into
// shared memory and every warp settles the remaining bits one at a time
// with ballots, without further barriers.
__device__ void fast_select(const ScoreArgs &a, FastSmem &fs, const float *srow,
                            const float (&c)[16], bool regs, int l0, unsigned kmax,
                            unsigned kmin, unsigned *K_out, int *need_out) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int need = a.cap_T;  // rank still to place among the keys matching prefix
    const unsigned diff = kmax ^ kmin;
    if (diff == 0u) {  // every key is the same value
        *K_out = kmax;
        *need_out = need;
        return;
    }
    int shift = (31 - __clz(int(diff))) & ~3;
    unsigned mask = shift >= 28 ? 0u : ~0u << (shift + 4);
    unsigned prefix = kmax & mask;
    int lo = 0, hi = l0;  // this request's keys that match prefix
    for (int pass = 0;; ++pass) {
        unsigned long long h0 = 0ull, h1 = 0ull;
        int nlo = hi, nhi = lo;
        if (regs) {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const unsigned key = __float_as_uint(c[k]);
                const bool v = k >= lo && k < hi && (key & mask) == prefix;
                count_digit(key, v, mask, prefix, shift, h0, h1);
                if (v) {
                    nlo = min(nlo, k);
                    nhi = k + 1;
                }
            }
        } else {
            for (int k = lo; k < hi; ++k) {
                const unsigned key = __float_as_uint(srow[k]);
                const bool v = (key & mask) == prefix;
                count_digit(key, v, mask, prefix, shift, h0, h1);
                if (v) {
                    nlo = min(nlo, k);
                    nhi = k + 1;
                }
            }
        }
        lo = nlo;
        hi = max(nhi, nlo);
        // bins 2q and 2q+1 as the 16-bit halves of word q
        const unsigned x0 = unsigned(h0), x1 = unsigned(h0 >> 32);
        const unsigned x2 = unsigned(h1), x3 = unsigned(h1 >> 32);
        unsigned w[8] = {__byte_perm(x0, 0u, 0x4140), __byte_perm(x0, 0u, 0x4342),
                         __byte_perm(x1, 0u, 0x4140), __byte_perm(x1, 0u, 0x4342),
                         __byte_perm(x2, 0u, 0x4140), __byte_perm(x2, 0u, 0x4342),
                         __byte_perm(x3, 0u, 0x4140), __byte_perm(x3, 0u, 0x4342)};
        unsigned (&wh)[kWarps][8] = fs.wh[pass & 1];
#pragma unroll
        for (int q = 0; q < 8; ++q) w[q] = __reduce_add_sync(0xffffffffu, w[q]);
        if (lane == 0) {
#pragma unroll
            for (int q = 0; q < 8; ++q) wh[warp][q] = w[q];
        }
        sync256();
        // lane t < 16 owns digit t: keys with digit >= t by a suffix scan
        unsigned cnt = 0u;
        if (lane < 16) {
#pragma unroll
            for (int v = 0; v < kWarps; ++v) cnt += wh[v][lane >> 1];
            cnt = (lane & 1) ? cnt >> 16 : cnt & 0xffffu;
        }
        unsigned suf = cnt;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
            const unsigned n = __shfl_down_sync(0xffffffffu, suf, o);
            if (lane + o < 16) suf += n;
        }
        const unsigned gt = suf - cnt;  // keys with a larger digit
        const unsigned hit = __ballot_sync(0xffffffffu, lane < 16 && gt < unsigned(need) &&
                                                            unsigned(need) <= suf);
        const int d = __ffs(int(hit)) - 1;  // exactly one lane holds the rank
        need -= int(__shfl_sync(0xffffffffu, gt, d));
        const int m = int(__shfl_sync(0xffffffffu, cnt, d));  // keys with digit d
        prefix |= unsigned(d) << shift;
        mask |= 15u << shift;
        if (shift == 0) break;
        if (m <= 32) {
            // Gather the m keys that match prefix (a warp scan of each
            // thread's count, one shared add per warp for its base).
            int mine = 0;
            if (regs) {
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    mine += k >= lo && k < hi && (__float_as_uint(c[k]) & mask) == prefix;
            } else {
                for (int k = lo; k < hi; ++k) mine += (__float_as_uint(srow[k]) & mask) == prefix;
            }
            int incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            int base = 0;
            if (lane == 31 && incl > 0) base = atomicAdd(&fs.ncand, incl);
            base = __shfl_sync(0xffffffffu, base, 31) + incl - mine;
            if (mine > 0) {
                if (regs) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const unsigned key = __float_as_uint(c[k]);
                        if (k >= lo && k < hi && (key & mask) == prefix) fs.cand[base++] = key;
                    }
                } else {
                    for (int k = lo; k < hi; ++k) {
                        const unsigned key = __float_as_uint(srow[k]);
                        if ((key & mask) == prefix) fs.cand[base++] = key;
                    }
                }
            }
            sync256();
            // Every warp settles the remaining bits from the same m keys.
            const unsigned key = lane < m ? fs.cand[lane] : 0u;
            for (int bit = shift - 1; bit >= 0; --bit) {
                const unsigned ones = unsigned(__popc(int(__ballot_sync(
                    0xffffffffu, lane < m && (key & mask) == prefix && ((key >> bit) & 1u)))));
                if (unsigned(need) <= ones) prefix |= 1u << bit;
                else need -= int(ones);
                mask |= 1u << bit;
            }
            break;
        }
        shift -= 4;
    }
    *K_out = prefix;
    *need_out = need;
}

__device__ void finish_fast(const ScoreArgs &a, uint8_t *ring) {
    __shared__ FastSmem fs;
    const int B = a.B, g = a.gamma, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pitch = g | 1;
    const FastLayout f = fast_layout(B, g, a.pack);
    int *ri = reinterpret_cast<int *>(ring);
    float *keys = reinterpret_cast<float *>(ring);
    const int b = tid;
    const bool own = b < B;
    float *srow = keys + b * pitch;
    if (tid == 0) fs.ncand = 0;  // ordered before its use by the barriers between

    // Survival curve and L0 of request b, 16 positions at a time.  S does
    // not increase with k (each factor is at most 1 and rounding is
    // monotone), so the k >= 1 with S_k >= c are exactly 1..L0_b.  The
    // first 16 confidences are loaded before the packing inputs are staged,
    // so that both sets of loads are in flight together.
    int l0 = 0;
    unsigned kfirst = 0u, klast = ~0u;
    const bool vec = (g & 3) == 0 &&
                     ((reinterpret_cast<uintptr_t>(a.conf) |
                       reinterpret_cast<uintptr_t>(a.survival)) & 15) == 0;
    const float *crow = a.conf + size_t(own ? b : 0) * g;
    float *orow = a.survival + size_t(own ? b : 0) * g;
    float c[16];
    load_conf16(crow, 0, own ? g : 0, vec, c);
    if (a.pack) {
        const int ntok = B * g;
        int tv[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int i = j * kThreads + tid;
            tv[j] = i < ntok ? __ldg(a.draft_tokens + i) : 0;
        }
        const int lt = own && a.last_tokens ? __ldg(a.last_tokens + b) : -1;
        const int sq = own && a.seq_lens ? __ldg(a.seq_lens + b) : 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int i = j * kThreads + tid;
            if (i < ntok) ri[f.tok + i] = tv[j];
        }
        if (own) {
            ri[f.last + b] = lt;
            ri[f.seq + b] = sq;
        }
        if (ntok > 16 * kThreads)
            stage_ints(ri + f.tok + 16 * kThreads, a.draft_tokens + 16 * kThreads,
                       ntok - 16 * kThreads);
    }
    if (own) {
        float S = 1.f;
        for (int k0 = 0; k0 < g; k0 += 16) {
            if (k0 > 0) load_conf16(crow, k0, g, vec, c);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (k0 + j < g) {
                    S *= c[j];
                    c[j] = S;
                    srow[k0 + j] = S;
                    l0 += S >= a.cost_c;
                }
            }
            if (vec) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (k0 + 4 * q < g)
                        reinterpret_cast<float4 *>(orow + k0)[q] =
                            make_float4(c[4 * q], c[4 * q + 1], c[4 * q + 2], c[4 * q + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (k0 + j < g) orow[k0 + j] = c[j];
            }
        }
        a.L0[b] = l0;
        if (l0 > 0) {
            kfirst = __float_as_uint(srow[0]);
            klast = __float_as_uint(srow[l0 - 1]);
        }
    }

    // sum L0, largest and smallest key
    {
        const int ws = __reduce_add_sync(0xffffffffu, l0);
        const unsigned wmax = __reduce_max_sync(0xffffffffu, kfirst);
        const unsigned wmin = __reduce_min_sync(0xffffffffu, klast);
        if (lane == 0) {
            fs.red[warp][0] = ws;
            fs.red[warp][1] = int(wmax);
            fs.red[warp][2] = int(wmin);
        }
    }
    sync256();
    int total = 0;
    unsigned kmax = 0u, kmin = ~0u;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        total += fs.red[w][0];
        kmax = max(kmax, unsigned(fs.red[w][1]));
        kmin = min(kmin, unsigned(fs.red[w][2]));
    }

    int L = l0;
    if (a.cap_T >= 0 && total > a.cap_T) {
        if (a.cap_T == 0) {
            L = 0;
        } else {
            unsigned K;
            int need;
            const bool regs = g <= 16;
            fast_select(a, fs, srow, c, regs, l0, kmax, kmin, &K, &need);
            // Keys above K are kept; of those equal to K, the first `need`
            // in (b, k) order.
            int above = 0, equal = 0;
            if (regs) {
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const unsigned key = __float_as_uint(c[k]);
                    above += k < l0 && key > K;
                    equal += k < l0 && key == K;
                }
            } else {
                for (int k = 0; k < l0; ++k) {
                    const unsigned key = __float_as_uint(srow[k]);
                    above += key > K;
                    equal += key == K;
                }
            }
            int tot_eq;
            const int ex = block_excl_scan_int(equal, &tot_eq, fs.sh);
            L = above + min(max(need - ex, 0), equal);
        }
    }

    // Offsets (the scan's barriers also retire every read of the keys).
    int tot_L;
    const int ex = block_excl_scan_int(L, &tot_L, fs.sh);
    if (own) {
        a.L[b] = L;
        a.draft_off[b] = ex;
        a.row_off[b] = ex + b;
    }
    if (tid == 0) {
        a.draft_off[B] = tot_L;
        a.row_off[B] = tot_L + B;
    }
    if (!a.pack) return;

    // Packing: the request of every packed row into shared memory, then
    // the four packed arrays written row by row.
    const int cap = B * (g + 1), n_rows = tot_L + B;
    if (own) {
        ri[f.roff + b] = ex + b;
        for (int j = 0; j <= L; ++j) ri[ex + b + j] = b;
    }
    sync256();
#pragma unroll 4
    for (int r = tid; r < n_rows; r += kThreads) {
        const int rb = ri[r], j = r - ri[f.roff + rb];
        a.packed_ids[r] = j == 0 ? ri[f.last + rb] : ri[f.tok + rb * g + j - 1];
        a.packed_pos[r] = ri[f.seq + rb] + j;
        a.row_req[r] = rb;
        a.row_k[r] = j;
    }
#pragma unroll 4
    for (int r = n_rows + tid; r < cap; r += kThreads) {
        a.packed_ids[r] = -1;
        a.packed_pos[r] = 0;
        a.row_req[r] = -1;
        a.row_k[r] = -1;
    }
}

__device__ void finish_batch(const ScoreArgs &a, uint8_t *ring) {
    if (fast_finish_fits(a)) finish_fast(a, ring);
    else finish_general(a, ring);
}

// Steps a1-a3: streaming confidence head (or, with kEntropy, the entropy of
// each draft row), survival curve, pre-cap lengths, then (in the CTA that
// finishes the batch) the cap and the scans.
template <typename T, bool kEntropy>
__device__ __forceinline__ void score_main(const ScoreArgs &a) {
    extern __shared__ __align__(1024) uint8_t ring[];
    __shared__ ScoreSmem sm;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid < kScoreStages) {
        mbar_init(&sm.full[tid], 1);
        mbar_init(&sm.empty[tid], kWarps);
        sm.done[tid] = 0;
    }
    if (tid == 0) {
        sm.run_cap = 0;
        fence_barrier_init();
    }
    if (a.pack) {
        // Only the finishing CTA reads the packing inputs, at the end: bring
        // them into L2 now, one 128-byte line per thread across the grid.
        const size_t line = size_t(blockIdx.x) * kScoreThreads + tid;
        const size_t tok_lines = (size_t(a.B) * a.gamma * 4 + 127) / 128;
        const size_t req_lines = (size_t(a.B) * 4 + 127) / 128;
        if (line < tok_lines) prefetch_l2(a.draft_tokens + line * 32);
        else if (line < tok_lines + req_lines && a.last_tokens)
            prefetch_l2(a.last_tokens + (line - tok_lines) * 32);
        else if (line < tok_lines + 2 * req_lines && a.seq_lens)
            prefetch_l2(a.seq_lens + (line - tok_lines - req_lines) * 32);
    }
    __syncthreads();
    const RowShape rs = row_shape(a, int(sizeof(T)));
    if (warp == kWarps) {
        if (lane == 0) score_producer(a, sm, ring, rs);
        return;
    }
    const int nrows = kEntropy ? entropy_consumer<T>(a, sm, ring, rs, warp, lane)
                               : score_consumer<T>(a, sm, ring, rs, warp, lane);
    // Publish this CTA's confidences; the CTA that adds the batch's last
    // rows finishes every request and runs the cap.  The barrier orders
    // every warp's confidence stores before thread 0's release fence and
    // count; the finishing CTA's thread 0 fences again (acquire) before the
    // barrier that lets its warps read every CTA's confidences from L2.
    sync256();
    if (tid == 0) {
        __threadfence();
        sm.run_cap = atomicAdd(a.done_cnt, nrows) + nrows == rs.rows;
        if (sm.run_cap) __threadfence();
    }
    sync256();
    if (!sm.run_cap) return;
    // Let the next kernel on the stream (the compaction or the verify, a
    // programmatic dependent launch) be scheduled now: every other CTA has
    // exited, so its CTAs take the freed slots in order.  It waits for this
    // grid to complete before it reads anything.  (Triggered at the start of
    // the kernel instead, its CTAs took slots as streaming CTAs exited and
    // the verify ran ~5 us slower.)
    asm volatile("griddepcontrol.launch_dependents;");
    finish_batch(a, ring);
    if (tid == 0) {
        *a.done_cnt = 0;
        *a.row_ctr = 0;
    }
}

template <typename T>
__global__ void __launch_bounds__(kScoreThreads, 3) score_budget_kernel(const ScoreArgs a) {
    score_main<T, false>(a);
}

template <typename T>
__global__ void __launch_bounds__(kScoreThreads, 3) score_entropy_kernel(const ScoreArgs a) {
    score_main<T, true>(a);
}

__global__ void __launch_bounds__(kThreads) fixed_budget_kernel(const FixedArgs a) {
    __shared__ int sh[kWarps + 1];
    asm volatile("griddepcontrol.launch_dependents;");
    const int l = a.F < a.gamma ? a.F : a.gamma;
    for (int b = threadIdx.x; b < a.B; b += kThreads) a.L[b] = l;
    __syncthreads();
    write_offsets(a.B, a.L, a.draft_off, a.row_off, sh);
}

// Fixed budget with the packing (steps a3 and a4 of the fixed mode): every
// L_b = l = min(F, gamma), so draft_off[b] = b * l and row_off[b] =
// b * (l + 1) in closed form and every slot is independent: one thread per
// slot (b, j) of the B*(gamma+1) capacity, as in the compaction kernel.
__global__ void __launch_bounds__(kThreads) fixed_pack_kernel(const FixedArgs a) {
    asm volatile("griddepcontrol.launch_dependents;");
    const int l = a.F < a.gamma ? a.F : a.gamma;
    const int g1 = a.gamma + 1, cap = a.B * g1, n_rows = a.B * (l + 1);
    const int t = blockIdx.x * kThreads + threadIdx.x;
    if (t <= a.B) {
        if (t < a.B) a.L[t] = l;
        a.draft_off[t] = t * l;
        a.row_off[t] = t * (l + 1);
    }
    if (t >= cap) return;
    const int b = t / g1, j = t - b * g1;
    if (j <= l) {
        const int r = b * (l + 1) + j;
        a.packed_ids[r] = j == 0 ? (a.last_tokens ? a.last_tokens[b] : -1)
                                 : a.draft_tokens[size_t(b) * a.gamma + j - 1];
        a.packed_pos[r] = (a.seq_lens ? a.seq_lens[b] : 0) + j;
        a.row_req[r] = b;
        a.row_k[r] = j;
    }
    if (t >= n_rows) {
        a.packed_ids[t] = -1;
        a.packed_pos[t] = 0;
        a.row_req[t] = -1;
        a.row_k[t] = -1;
    }
}

}  // namespace

template <bool kEntropy>
static int blocks_per_sm(int bf16) {
    const int bytes = int(kScoreSmemBytes);
    void (*kern)(const ScoreArgs) =
        kEntropy ? (bf16 ? score_entropy_kernel<uint16_t> : score_entropy_kernel<float>)
                 : (bf16 ? score_budget_kernel<uint16_t> : score_budget_kernel<float>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return -1;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kScoreThreads, kScoreSmemBytes);
    return e == cudaSuccess ? n : -1;
}

int score_blocks_per_sm(int hidden_bf16) { return blocks_per_sm<false>(hidden_bf16); }

int entropy_blocks_per_sm(int logit_bf16) { return blocks_per_sm<true>(logit_bf16); }

cudaError_t launch_score_budget(const ScoreArgs &a, int grid, cudaStream_t s) {
    if (a.hidden_bf16)
        score_budget_kernel<uint16_t><<<grid, kScoreThreads, kScoreSmemBytes, s>>>(a);
    else
        score_budget_kernel<float><<<grid, kScoreThreads, kScoreSmemBytes, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_score_entropy(const ScoreArgs &a, int grid, cudaStream_t s) {
    if (a.hidden_bf16)
        score_entropy_kernel<uint16_t><<<grid, kScoreThreads, kScoreSmemBytes, s>>>(a);
    else
        score_entropy_kernel<float><<<grid, kScoreThreads, kScoreSmemBytes, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fixed_budget(const FixedArgs &a, cudaStream_t s) {
    if (a.pack) {
        const long long slots = std::max<long long>((long long)a.B * (a.gamma + 1), a.B + 1LL);
        fixed_pack_kernel<<<int((slots + kThreads - 1) / kThreads), kThreads, 0, s>>>(a);
    } else {
        fixed_budget_kernel<<<1, kThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace dspark
