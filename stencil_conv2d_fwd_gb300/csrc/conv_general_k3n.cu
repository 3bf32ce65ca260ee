// Direct convolution for kernel size K = 3, 16 or fewer output channels.
#include "conv_general.cuh"

namespace sc {
// Small images with up to 16 input channels take the whole-tile kernel
// (conv_small.cu), the rest the TMA-staged kernel (conv_tma_k3.cu), and
// these cp.async-staged configurations where neither applies.
cudaError_t launch_conv_general_k3_narrow(const ConvArgs &a, cudaStream_t st)
{
    cudaError_t e = launch_conv_small(a, st);
    if (e != cudaErrorNotSupported) return e;
    e = launch_conv_tma_k3_narrow(a, st);
    if (e != cudaErrorNotSupported) return e;
    return dispatch_narrow<3, 8>(a, st);
}
}  // namespace sc
