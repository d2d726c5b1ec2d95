// sts_fit.cu -- fitting the STS temperatures to logged accept outcomes.
//
// "DFlash to DSpark in SGLang", section "DSpark: a sequential head and a
// verify budget": Sequential Temperature Scaling calibrates the head's
// survival product to match true acceptance rates.  Position i's temperature
// tau_i in conf = sigmoid(x / tau_i) is fitted by maximum likelihood on
// logged steps.  A logged request-step n (verify length L_n, accepted drafts
// a_n) observes position i when i < L_n and i <= a_n; the outcome y is 1 for
// an accept (i < a_n) and 0 for the first rejection (i = a_n).  The head
// logit comes back from the logged confidence and the temperature that
// produced it, x = tau_used_i * logit(conf), with conf clamped to
// [2^-126, 1 - 2^-24], the range of an fp32 confidence below 1.
//
// With beta = 1 / tau the negative log-likelihood
//   NLL(beta) = sum_obs log(1 + e^{beta x}) - y beta x
// is convex, and its derivative g(beta) = sum_obs x (sigmoid(beta x) - y)
// does not decrease.  One CTA per position bisects [1/tau_max, 1/tau_min]
// on the sign of g (a minimum on a bound when g keeps one sign there).
// Terms are fp32, sums fp64, reduced in a fixed order: the fit is
// deterministic.  This is offline calibration over the logs, not a step of
// the per-step path.
#include "dspark_internal.cuh"
#include "sts_fit.cuh"

namespace dspark {
namespace {

constexpr int kFitThreads = kThreads;  // 8 warps
constexpr int kFitBisections = 60;

// Sum of one double per thread over the CTA, the same in every thread.
__device__ double cta_sum(double v, double *sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    double t = 0.0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += sh[w];
    __syncthreads();
    return t;
}

__device__ __forceinline__ bool observed(const FitArgs &a, int n, int i, int *y) {
    const int L = a.L[n], acc = a.accept_len[n];
    *y = i < acc;
    return i < L && i <= acc;
}

__device__ __forceinline__ float logit_of(const FitArgs &a, int n, int i, float tu) {
    float c = a.conf[size_t(n) * a.gamma + i];
    c = fminf(fmaxf(c, 1.17549435e-38f), 0.99999994f);
    return tu * (logf(c) - log1pf(-c));
}

// g(beta) = sum_obs x (sigmoid(beta x) - y)
__device__ double grad(const FitArgs &a, int i, float tu, double beta, double *sh) {
    double s = 0.0;
    const float b = float(beta);
    for (int n = threadIdx.x; n < a.N; n += kFitThreads) {
        int y;
        if (!observed(a, n, i, &y)) continue;
        const float x = logit_of(a, n, i, tu);
        const float sg = 1.f / (1.f + expf(-b * x));
        s += double(x * (sg - float(y)));
    }
    return cta_sum(s, sh);
}

__global__ void __launch_bounds__(kFitThreads) sts_fit_kernel(const FitArgs a) {
    __shared__ double sh[kWarps];
    const int i = blockIdx.x;
    const float tu = a.tau_used[i];
    double cnt = 0.0;
    for (int n = threadIdx.x; n < a.N; n += kFitThreads) {
        int y;
        cnt += observed(a, n, i, &y) ? 1.0 : 0.0;
    }
    const int nobs = int(cta_sum(cnt, sh));
    if (nobs == 0) {
        if (threadIdx.x == 0) {
            a.tau_out[i] = tu;
            if (a.nll_out) a.nll_out[i] = 0.f;
            if (a.n_obs) a.n_obs[i] = 0;
        }
        return;
    }
    double lo = 1.0 / double(a.tau_max), hi = 1.0 / double(a.tau_min);
    double beta;
    if (grad(a, i, tu, hi, sh) <= 0.0) {
        beta = hi;
    } else if (grad(a, i, tu, lo, sh) >= 0.0) {
        beta = lo;
    } else {
        for (int it = 0; it < kFitBisections; ++it) {
            const double mid = 0.5 * (lo + hi);
            if (grad(a, i, tu, mid, sh) > 0.0) hi = mid;
            else lo = mid;
        }
        beta = 0.5 * (lo + hi);
    }
    double nll = 0.0;
    const float b = float(beta);
    for (int n = threadIdx.x; n < a.N; n += kFitThreads) {
        int y;
        if (!observed(a, n, i, &y)) continue;
        const float z = b * logit_of(a, n, i, tu);
        const float sp = z > 0.f ? z + log1pf(expf(-z)) : log1pf(expf(z));
        nll += double(sp) - (y ? double(z) : 0.0);
    }
    nll = cta_sum(nll, sh);
    if (threadIdx.x == 0) {
        a.tau_out[i] = float(1.0 / beta);
        if (a.nll_out) a.nll_out[i] = float(nll);
        if (a.n_obs) a.n_obs[i] = nobs;
    }
}

}  // namespace

cudaError_t launch_sts_fit(const FitArgs &a, cudaStream_t s) {
    sts_fit_kernel<<<a.gamma, kFitThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace dspark
