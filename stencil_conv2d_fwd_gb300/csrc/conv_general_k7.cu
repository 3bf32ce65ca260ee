// Instantiations of the general direct convolution for kernel size K = 7
// (filters up to 7x7, centred).
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_k7(const ConvArgs &a, cudaStream_t st) { return dispatch_general<7>(a, st); }
}  // namespace sc
