// Diagnostics that measure the hardware the attention kernels run on, rather
// than compute attention: a throughput microbenchmark of the exponential
// unit, the second bound of the forward and backward kernels after the tensor
// core (one 2^x per score element).
#include <cuda_runtime.h>

#include "fa_internal.h"

namespace fa {
namespace {

// Every thread runs eight independent chains x <- 2^(-x) of
// ex2.approx.ftz.f32 for `iters` rounds (the values stay in [1/2, 1]) and
// stores their sum, so that every exp is live.  With eight blocks of 256
// threads an SM the unit, not the chains' latency, sets the time.
__global__ void __launch_bounds__(256) fa_ex2_rate_kernel(float* __restrict__ out, int iters) {
    float x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = 0.25f + 0.0625f * k + 1e-7f * threadIdx.x;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = ex2(-x[k]);
    }
    float sum = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) sum += x[k];
    out[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = sum;
}

}  // namespace

cudaError_t launch_ex2_rate(float* out, int blocks, int iters, cudaStream_t stream) {
    count_launch();
    fa_ex2_rate_kernel<<<blocks, 256, 0, stream>>>(out, iters);
    return cudaGetLastError();
}

}  // namespace fa
