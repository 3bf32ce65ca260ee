// Instantiations of the general direct convolution for kernel size K = 5
// (filters up to 5x5, centred).
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_k5(const ConvArgs &a, cudaStream_t st)
{
    constexpr int CS = stage_channels_small<5>();
    return a.Cout > 16 ? dispatch_wide<5, CS>(a, st) : dispatch_narrow<5, CS>(a, st);
}
}  // namespace sc
