// Direct convolution for kernel size K = 5
// (filters up to 5x5, centred).
#include "conv_general.cuh"

namespace sc {
// 16 or fewer output channels: the TMA-staged kernel (conv_tma_k5.cu) first
// (32 -> 4 on 1280 x 720: 127 us against 165 us); more channels and filter
// banks above its limit: these cp.async-staged configurations (32 -> 32:
// 798 us against 824 us for the TMA kernel; 25 taps per staged pixel make
// the staging cost small; the TMA kernel with 5 or 7 pixels per thread
// measured 806-824 us).
cudaError_t launch_conv_general_k5(const ConvArgs &a, cudaStream_t st)
{
    if (a.Cout <= 16) {
        const cudaError_t e = launch_conv_tma_k5_narrow(a, st);
        if (e != cudaErrorNotSupported) return e;
    }
    constexpr int CS = stage_channels_small<5>();
    return a.Cout > 16 ? dispatch_wide<5, CS>(a, st) : dispatch_narrow<5, CS>(a, st);
}
}  // namespace sc
