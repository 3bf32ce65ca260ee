// Instantiations of the general direct convolution for kernel size K = 3
// (filters up to 3x3, centred).
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_k3(const ConvArgs &a, cudaStream_t st) { return dispatch_general<3>(a, st); }
}  // namespace sc
