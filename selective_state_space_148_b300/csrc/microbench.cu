// microbench.cu -- throughput of ex2.approx.ftz.f32 on the special-function
// (MUFU) pipe.  The scan issues one such exp per (b, d, n, t), so this rate,
// not FMA throughput, is the compute roofline the scan is measured against.
// Each thread runs 8 independent dependency chains so that issue, not
// latency, limits the rate; each CTA reports its elapsed SM clocks.
#include "internal.h"

namespace mamba {

__global__ void bench_ex2_kernel(long long *cycles, float *sink, long long iters) {
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = -0.001f * (float)(threadIdx.x + j);
    __syncthreads();
    const long long t0 = clock64();
    for (long long it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = ex2_approx(x[j]) - 1.0f;  // stays in (-1, 0]
    }
    __syncthreads();
    const long long t1 = clock64();
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc += x[j];
    sink[(long long)blockIdx.x * blockDim.x + threadIdx.x] = acc;
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

cudaError_t launch_bench_ex2(long long *cycles, float *sink, long long iters, int blocks, int threads,
                             cudaStream_t st) {
    bench_ex2_kernel<<<blocks, threads, 0, st>>>(cycles, sink, iters);
    return cudaGetLastError();
}

}  // namespace mamba
