// Instantiations of the general direct convolution for S = 3 taps per row.
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_s3(const ConvArgs &a, cudaStream_t st) { return dispatch_general<3>(a, st); }
}  // namespace sc
