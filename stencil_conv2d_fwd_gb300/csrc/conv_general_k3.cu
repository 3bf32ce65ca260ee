// Instantiations of the general direct convolution for kernel size K = 3,
// more than 16 output channels (conv_general_k3n.cu has the rest).
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_k3_narrow(const ConvArgs &a, cudaStream_t st);

cudaError_t launch_conv_general_k3(const ConvArgs &a, cudaStream_t st)
{
    if (a.Cout <= 16) return launch_conv_general_k3_narrow(a, st);
    if (a.Cin % 16 == 0) return dispatch_wide<3, 16>(a, st);
    return dispatch_wide<3, 8>(a, st);
}
}  // namespace sc
