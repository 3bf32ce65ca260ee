// Direct convolution for kernel size K = 1
// (filters up to 1x1, centred).
#include "conv_general.cuh"

namespace sc {
// The TMA-staged kernel (conv_tma_k1.cu) first; these cp.async-staged
// configurations where it does not apply (filter banks above its limit).
cudaError_t launch_conv_general_k1(const ConvArgs &a, cudaStream_t st)
{
    const cudaError_t e = a.Cout > 16 ? launch_conv_tma_k1_wide(a, st) : launch_conv_tma_k1_narrow(a, st);
    if (e != cudaErrorNotSupported) return e;
    constexpr int CS = stage_channels_small<1>();
    return a.Cout > 16 ? dispatch_wide<1, CS>(a, st) : dispatch_narrow<1, CS>(a, st);
}
}  // namespace sc
