// Instantiations of the general direct convolution for kernel size K = 1
// (filters up to 1x1, centred).
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_k1(const ConvArgs &a, cudaStream_t st)
{
    constexpr int CS = stage_channels_small<1>();
    return a.Cout > 16 ? dispatch_wide<1, CS>(a, st) : dispatch_narrow<1, CS>(a, st);
}
}  // namespace sc
