// Instantiations of the general direct convolution for S = 5 taps per row.
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_s5(const ConvArgs &a, cudaStream_t st) { return dispatch_general<5>(a, st); }
}  // namespace sc
