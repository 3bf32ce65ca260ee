// Instantiations of the general direct convolution for kernel size K = 1
// (filters up to 1x1, centred).
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_k1(const ConvArgs &a, cudaStream_t st) { return dispatch_general<1>(a, st); }
}  // namespace sc
