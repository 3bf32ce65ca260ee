// Instantiations of the general direct convolution for S = 7 taps per row.
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_s7(const ConvArgs &a, cudaStream_t st) { return dispatch_general<7>(a, st); }
}  // namespace sc
