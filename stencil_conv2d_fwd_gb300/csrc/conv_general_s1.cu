// Instantiations of the general direct convolution for S = 1 taps per row.
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_s1(const ConvArgs &a, cudaStream_t st) { return dispatch_general<1>(a, st); }
}  // namespace sc
