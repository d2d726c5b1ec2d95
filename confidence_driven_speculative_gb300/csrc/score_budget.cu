// score_budget.cu -- steps a1-a3 and the scans of a4 in one kernel.
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
// by request then position, followed by the exclusive scans.  Counters reset
// themselves, so no CTA waits on another and the kernel is safe to replay.
//
// score_entropy_kernel is the same kernel with the draft logit rows as its
// rows and an entropy consumer in place of the dot product: the confidence of
// a draft is exp(-H) of its distribution ("SGLang Integrates DSpark ...",
// "DSpark's Core Idea: Only Verify the Parts You're Confident About").
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
    float tau[DSPARK_MAX_GAMMA];       // STS temperatures
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
        if (r < rs.rows) next = int(gridDim.x) + atomicAdd(a.row_ctr, 1);
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
        // The row's bias is needed at its end; load it now, behind the FMAs.
        const int rb = r / a.gamma;
        const float bias = q + 1 == rs.ntr ? __ldg(&a.head_bias[rb]) : 0.f;
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
            const float x = (dot + bias) / sm.tau[r - rb * a.gamma];
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

__device__ void finish_and_budget(const ScoreArgs &a, uint8_t *ring) {
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
}

// Steps a1-a3: streaming confidence head (or, with kEntropy, the entropy of
// each draft row), survival curve, pre-cap lengths, then (in the CTA that
// finishes the batch) the cap and the scans.
template <typename T, bool kEntropy>
__device__ __forceinline__ void score_main(const ScoreArgs &a) {
    extern __shared__ __align__(1024) uint8_t ring[];
    __shared__ ScoreSmem sm;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Let the next kernel on the stream (the compaction, a programmatic
    // dependent launch) be scheduled now; it waits for this grid to complete
    // before it reads anything.
    asm volatile("griddepcontrol.launch_dependents;");
    if (tid < kScoreStages) {
        mbar_init(&sm.full[tid], 1);
        mbar_init(&sm.empty[tid], kWarps);
        sm.done[tid] = 0;
    }
    if (tid == 0) {
        sm.run_cap = 0;
        fence_barrier_init();
    }
    if (!kEntropy && tid < a.gamma) sm.tau[tid] = a.sts_tau[tid];
    __syncthreads();
    const RowShape rs = row_shape(a, int(sizeof(T)));
    if (warp == kWarps) {
        if (lane == 0) score_producer(a, sm, ring, rs);
        return;
    }
    const int nrows = kEntropy ? entropy_consumer<T>(a, sm, ring, rs, warp, lane)
                               : score_consumer<T>(a, sm, ring, rs, warp, lane);
    // Publish this CTA's confidences; the CTA that adds the batch's last
    // rows finishes every request and runs the cap.
    __threadfence();
    sync256();
    if (tid == 0) sm.run_cap = atomicAdd(a.done_cnt, nrows) + nrows == rs.rows;
    sync256();
    if (!sm.run_cap) return;
    __threadfence();
    finish_and_budget(a, ring);
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
    const int l = a.F < a.gamma ? a.F : a.gamma;
    for (int b = threadIdx.x; b < a.B; b += kThreads) a.L[b] = l;
    __syncthreads();
    write_offsets(a.B, a.L, a.draft_off, a.row_off, sh);
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
    fixed_budget_kernel<<<1, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace dspark
