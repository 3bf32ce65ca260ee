// Instantiations of the narrow-output convolution (conv_narrow.cuh): 3 x 3
// filters, 4 output channels, 32 input channels.
#include "autotune.h"
#include "conv_narrow.cuh"

namespace sc {

// <W_T, tile rows, channels a step, stages, CTAs per SM, steps per tile>
cudaError_t k3_n4_h8_s4(const ConvArgs &a, cudaStream_t st) { return launch_conv_n4<N4Cfg<5, 8, 8, 4, 1, 4>>(a, st); }
cudaError_t k3_n4_h8_c16(const ConvArgs &a, cudaStream_t st) { return launch_conv_n4<N4Cfg<5, 8, 16, 2, 1, 2>>(a, st); }

}  // namespace sc
