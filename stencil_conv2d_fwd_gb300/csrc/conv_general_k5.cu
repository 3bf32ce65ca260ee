// Instantiations of the general direct convolution for kernel size K = 5
// (filters up to 5x5, centred).
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_k5(const ConvArgs &a, cudaStream_t st) { return dispatch_general<5>(a, st); }
}  // namespace sc
