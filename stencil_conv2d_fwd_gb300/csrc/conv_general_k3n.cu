// Instantiations of the general direct convolution for kernel size K = 3,
// 16 or fewer output channels.
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_k3_narrow(const ConvArgs &a, cudaStream_t st) { return dispatch_narrow<3, 8>(a, st); }
}  // namespace sc
