// Direct convolution for kernel size K = 3, 16 or fewer output channels.
#include "conv_general.cuh"

namespace sc {
// The TMA-staged kernel first (conv_tma_k3.cu); these cp.async-staged
// configurations where it does not apply.
cudaError_t launch_conv_general_k3_narrow(const ConvArgs &a, cudaStream_t st)
{
    const cudaError_t e = launch_conv_tma_k3_narrow(a, st);
    if (e != cudaErrorNotSupported) return e;
    return dispatch_narrow<3, 8>(a, st);
}
}  // namespace sc
