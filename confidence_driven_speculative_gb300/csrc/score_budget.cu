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
// Work split.  Grid = B x splits CTAs of 256 threads.  CTA (b, s) streams the
// s-th slice of the d-vector of every draft position of request b (16-byte
// loads, one warp per position, fp32 FMAs) and writes partial dot products.
// The last CTA of request b (per-request counter) sums the slices in a fixed
// order, applies bias, 1/tau_i and the sigmoid, forms the cumulative product
// S and the pre-cap length L0_b.  The last request to finish (batch counter)
// runs the cap in that one CTA: an MSB-first radix select over the fp32 bit
// patterns of the candidate gains S_{b,k} (non-negative floats order like
// their bit patterns), ties resolved by request then position, followed by
// the exclusive scans.  Counters reset themselves, so nothing waits and the
// kernel is safe to replay.
#include "dspark_internal.cuh"

namespace dspark {
namespace {

// Block-wide exclusive scan of one int per thread; *total gets the sum.
// `sh` needs kWarps + 1 ints.  Contains __syncthreads.
__device__ int block_excl_scan_int(int v, int *total, int *sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int x = lane < kWarps ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += n;
        }
        if (lane < kWarps) sh[lane] = x;
    }
    __syncthreads();
    const int before = warp > 0 ? sh[warp - 1] : 0;
    *total = sh[kWarps - 1];
    __syncthreads();
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

// The cap, run by one CTA once every L0 and S of the batch is written.
constexpr int kSmemKeys = 4096;  // candidate keys the cap stages in shared memory

__device__ void budget_and_scan(const ScoreArgs &a) {
    __shared__ unsigned keys[kSmemKeys];
    __shared__ int sh[kWarps + 1];
    __shared__ unsigned hist[256];
    __shared__ int sel[2];
    const int B = a.B, g = a.gamma, tid = threadIdx.x;

    int part = 0;
    for (int b = tid; b < B; b += kThreads) part += __ldcg(&a.L0[b]);
    int sum;
    block_excl_scan_int(part, &sum, sh);

    if (a.cap_T < 0 || sum <= a.cap_T) {
        for (int b = tid; b < B; b += kThreads) a.L[b] = __ldcg(&a.L0[b]);
    } else if (a.cap_T == 0) {
        for (int b = tid; b < B; b += kThreads) a.L[b] = 0;
    } else {
        // Find the cap_T-th largest candidate key, 8 bits per pass from the top.
        // Up to kSmemKeys candidate keys are staged in shared memory (one
        // round of loads, non-candidates marked 0xffffffff); larger batches
        // are re-read from L2 each pass.
        const int nkeys = B * g;
        const bool staged = nkeys <= kSmemKeys;
        if (staged) {
            for (int f = tid; f < nkeys; f += kThreads) {
                const int b = f / g, k = f - b * g + 1;
                const int l0 = __ldcg(&a.L0[b]);
                const unsigned kv = __float_as_uint(__ldcg(&a.survival[f]));
                keys[f] = k <= l0 ? kv : 0xffffffffu;
            }
        }
        unsigned prefix = 0, mask = 0;
        int need = a.cap_T;  // rank still to place within keys matching `prefix`
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
            if (tid == 0) {
                sel[0] = 0;
                sel[1] = need;
            }
            __syncthreads();
            if (staged) {
                for (int f = tid; f < nkeys; f += kThreads) {
                    const unsigned kv = keys[f];
                    if (kv != 0xffffffffu && (kv & mask) == prefix)
                        atomicAdd(&hist[(kv >> shift) & 255u], 1u);
                }
            } else {
                for (int f = tid; f < nkeys; f += kThreads) {
                    const int b = f / g, k = f - b * g + 1;
                    if (k <= __ldcg(&a.L0[b])) {
                        const unsigned kv = __float_as_uint(__ldcg(&a.survival[f]));
                        if ((kv & mask) == prefix) atomicAdd(&hist[(kv >> shift) & 255u], 1u);
                    }
                }
            }
            __syncthreads();
            if (tid < 32) {
                // lane l owns bins 8l .. 8l+7; suffix sums from the top bin down
                unsigned local = 0;
#pragma unroll
                for (int q = 0; q < 8; ++q) local += hist[tid * 8 + q];
                unsigned suf = local;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned n = __shfl_down_sync(0xffffffffu, suf, o);
                    if (tid + o < 32) suf += n;
                }
                const unsigned above = suf - local;  // keys in bins above this lane's
                const bool hit = above < unsigned(need) && unsigned(need) <= suf;
                if (hit) {
                    unsigned cum = above;
                    for (int q = 7; q >= 0; --q) {
                        const unsigned c = hist[tid * 8 + q];
                        if (cum + c >= unsigned(need)) {
                            sel[0] = tid * 8 + q;
                            sel[1] = need - int(cum);
                            break;
                        }
                        cum += c;
                    }
                }
            }
            __syncthreads();
            prefix |= unsigned(sel[0]) << shift;
            mask |= 255u << shift;
            need = sel[1];
            __syncthreads();
        }
        // prefix is the threshold key; `need` keys equal to it are kept, the
        // lowest (b, k) first.  Within a request keys do not increase with k,
        // so the kept set of each request is a prefix.
        int carry = 0;
        for (int base = 0; base < B; base += kThreads) {
            const int b = base + tid;
            int above = 0, equal = 0;
            if (b < B) {
                const int l0 = __ldcg(&a.L0[b]);
                for (int k = 1; k <= l0; ++k) {
                    const unsigned key = staged ? keys[b * g + k - 1]
                                                : __float_as_uint(__ldcg(&a.survival[b * g + k - 1]));
                    above += key > prefix;
                    equal += key == prefix;
                }
            }
            int total;
            const int ex = block_excl_scan_int(equal, &total, sh);
            if (b < B) {
                const int keep = min(max(need - (carry + ex), 0), equal);
                a.L[b] = above + keep;
            }
            carry += total;
        }
    }
    __syncthreads();
    write_offsets(B, a.L, a.draft_off, a.row_off, sh);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) score_budget_kernel(const ScoreArgs a) {
    constexpr int VE = Vec<T>::kElems;
    constexpr int U = 8;  // 16-byte loads in flight per lane and position
    __shared__ float4 w_s[kMaxSliceVec * VE / 4];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x / a.splits, s = blockIdx.x - b * a.splits;
    const int g = a.gamma;
    const int nvec = a.d / VE;
    const int v0 = int((long long)nvec * s / a.splits);
    const int v1 = int((long long)nvec * (s + 1) / a.splits);
    const int nv = v1 - v0;  // <= kMaxSliceVec (the host picks the splits)
    const float4 *w4 = reinterpret_cast<const float4 *>(a.head_w) + size_t(v0) * VE / 4;
    for (int i = tid; i < nv * VE / 4; i += kThreads) w_s[i] = __ldg(w4 + i);
    __syncthreads();

    // Warp w takes positions w, w + 8, ...; two at a time, their loads
    // interleaved so 2U loads per lane are in flight.
    for (int i0 = warp; i0 < g; i0 += 2 * kWarps) {
        const int i1 = i0 + kWarps;
        const bool two = i1 < g;
        const uint4 *h0 = reinterpret_cast<const uint4 *>(
            static_cast<const char *>(a.hidden) + (size_t(b) * g + i0) * size_t(a.d) * sizeof(T)) + v0;
        const uint4 *h1 = reinterpret_cast<const uint4 *>(
            static_cast<const char *>(a.hidden) + (size_t(b) * g + (two ? i1 : i0)) * size_t(a.d) * sizeof(T)) + v0;
        float acc0 = 0.f, acc1 = 0.f;
        for (int vb = 0; vb < nv; vb += 32 * U) {
            uint4 x0[U], x1[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = vb + lane + 32 * u;
                x0[u] = v < nv ? __ldcs(h0 + v) : make_uint4(0, 0, 0, 0);
                x1[u] = (two && v < nv) ? __ldcs(h1 + v) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = vb + lane + 32 * u;
                if (v < nv) {
                    float e0[VE], e1[VE];
                    Vec<T>::unpack(x0[u], e0);
                    Vec<T>::unpack(x1[u], e1);
#pragma unroll
                    for (int e = 0; e < VE; e += 4) {
                        const float4 wv = w_s[(v * VE + e) / 4];
                        acc0 = fmaf(e0[e], wv.x, acc0);
                        acc0 = fmaf(e0[e + 1], wv.y, acc0);
                        acc0 = fmaf(e0[e + 2], wv.z, acc0);
                        acc0 = fmaf(e0[e + 3], wv.w, acc0);
                        acc1 = fmaf(e1[e], wv.x, acc1);
                        acc1 = fmaf(e1[e + 1], wv.y, acc1);
                        acc1 = fmaf(e1[e + 2], wv.z, acc1);
                        acc1 = fmaf(e1[e + 3], wv.w, acc1);
                    }
                }
            }
        }
        acc0 = warp_sum(acc0);
        acc1 = warp_sum(acc1);
        if (lane == 0) {
            a.dot_part[(size_t(b) * g + i0) * kMaxScoreSplits + s] = acc0;
            if (two) a.dot_part[(size_t(b) * g + i1) * kMaxScoreSplits + s] = acc1;
        }
    }

    __shared__ int s_last;
    __shared__ float s_conf[DSPARK_MAX_GAMMA];
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(&a.req_cnt[b], 1) == a.splits - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // Last slice of request b: finish the head and the survival curve.
    if (tid < g) {
        float dot = 0.f;
        for (int q = 0; q < a.splits; ++q)
            dot += __ldcg(&a.dot_part[(size_t(b) * g + tid) * kMaxScoreSplits + q]);
        const float x = (dot + a.head_bias[b]) / a.sts_tau[tid];
        const float c = 1.f / (1.f + expf(-x));
        a.conf[size_t(b) * g + tid] = c;
        s_conf[tid] = c;
    }
    __syncthreads();
    if (tid == 0) {
        float S = 1.f;  // S_0
        int L = 1.f >= a.cost_c ? 0 : -1;
        for (int k = 1; k <= g; ++k) {
            S *= s_conf[k - 1];
            a.survival[size_t(b) * g + k - 1] = S;
            if (S >= a.cost_c) L = k;
        }
        a.L0[b] = L < 0 ? 0 : L;
        a.req_cnt[b] = 0;
        __threadfence();
        s_last = atomicAdd(a.done_cnt, 1) == a.B - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    budget_and_scan(a);
    if (tid == 0) *a.done_cnt = 0;
}

__global__ void __launch_bounds__(kThreads) fixed_budget_kernel(const FixedArgs a) {
    __shared__ int sh[kWarps + 1];
    const int l = a.F < a.gamma ? a.F : a.gamma;
    for (int b = threadIdx.x; b < a.B; b += kThreads) a.L[b] = l;
    __syncthreads();
    write_offsets(a.B, a.L, a.draft_off, a.row_off, sh);
}

}  // namespace

cudaError_t launch_score_budget(const ScoreArgs &a, int grid, cudaStream_t s) {
    if (a.hidden_bf16)
        score_budget_kernel<uint16_t><<<grid, kThreads, 0, s>>>(a);
    else
        score_budget_kernel<float><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fixed_budget(const FixedArgs &a, cudaStream_t s) {
    fixed_budget_kernel<<<1, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace dspark
