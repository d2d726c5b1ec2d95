// sts_fit.cuh -- argument block and launcher of the STS temperature fit.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dspark {

struct FitArgs {
    int N, gamma;
    const float *conf, *tau_used;
    const int32_t *L, *accept_len;
    float tau_min, tau_max;
    float *tau_out, *nll_out;
    int32_t *n_obs;
};

cudaError_t launch_sts_fit(const FitArgs &a, cudaStream_t s);

}  // namespace dspark
