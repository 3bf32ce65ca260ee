// Direct convolution for kernel size K = 3, more than 16 output channels
// (conv_general_k3n.cu has the rest).
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_k3_narrow(const ConvArgs &a, cudaStream_t st);

// The TMA-staged kernel (conv_tma_k3.cu) first; the cp.async-staged
// configurations where it does not apply (filter banks above its limit).
cudaError_t launch_conv_general_k3(const ConvArgs &a, cudaStream_t st)
{
    if (a.Cout <= 16) return launch_conv_general_k3_narrow(a, st);
    const cudaError_t e = launch_conv_tma_k3_wide(a, st);
    if (e != cudaErrorNotSupported) return e;
    if (a.Cin % 16 == 0) return dispatch_wide<3, 16>(a, st);
    return dispatch_wide<3, 8>(a, st);
}

// The wide configurations of dispatch_wide<3, 16>, one by one, for the
// autotuner (it must not instantiate them a second time elsewhere: each
// translation unit registers its own copy of a kernel, and the
// shared-memory opt-in of one copy does not reach the other).
cudaError_t k3_wide_w7_f64(const ConvArgs &a, cudaStream_t st) { return launch_gen_auto<3, 64, 7, 8, 28, 16, 1>(a, st); }
cudaError_t k3_wide_w8_f64(const ConvArgs &a, cudaStream_t st) { return launch_gen_auto<3, 64, 8, 8, 32, 16, 1>(a, st); }
cudaError_t k3_wide_w7_f32(const ConvArgs &a, cudaStream_t st) { return launch_gen_auto<3, 32, 7, 8, 56, 16, 1>(a, st); }
cudaError_t k3_wide_w8_f32(const ConvArgs &a, cudaStream_t st) { return launch_gen_auto<3, 32, 8, 8, 64, 16, 1>(a, st); }
}  // namespace sc
