// FP32 FMA rate probe: each thread runs 16 independent FMA chains, enough
// to cover the FMA latency with one warp per scheduler, so the issue rate
// of the FP32 pipes bounds the kernel.  Used to report the measured FP32
// FFMA peak beside the nominal one.
#include "common.cuh"
#include "launch.h"

namespace sc {

__global__ void __launch_bounds__(256) ffma_peak_kernel(float *sink, int iters)
{
    float a[16];
    const float m = 0.999999f, c = 1.0e-7f;
#pragma unroll
    for (int k = 0; k < 16; ++k) a[k] = 1.0f + 1.0e-3f * (threadIdx.x + k);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < 16; ++k) a[k] = fmaf(a[k], m, c);
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) s += a[k];
    sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// Launch-cost probe: a kernel that does nothing, so a run of it measures
// the floor of one launch (back to back, e.g. replayed from a CUDA graph).
__global__ void empty_kernel() {}

cudaError_t launch_empty(int blocks, int threads, cudaStream_t st)
{
    empty_kernel<<<blocks, threads, 0, st>>>();
    return cudaGetLastError();
}

cudaError_t launch_ffma_peak(float *sink, int blocks, int iters, cudaStream_t st)
{
    ffma_peak_kernel<<<blocks, 256, 0, st>>>(sink, iters);
    return cudaGetLastError();
}

}  // namespace sc
