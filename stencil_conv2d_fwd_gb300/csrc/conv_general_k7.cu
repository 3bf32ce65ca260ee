// Instantiations of the general direct convolution for kernel size K = 7
// (filters up to 7x7, centred).
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_k7(const ConvArgs &a, cudaStream_t st)
{
    constexpr int CS = stage_channels_small<7>();
    return a.Cout > 16 ? dispatch_wide<7, CS>(a, st) : dispatch_narrow<7, CS>(a, st);
}
}  // namespace sc
