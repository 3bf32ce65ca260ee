// Instantiations of the TMA-staged direct convolution (conv_tma.cuh) for
// 5 x 5 filters and 16 or fewer output channels.  A 5 x 5 tile stage carries
// 4 halo rows and columns, so these configurations keep two stages to fit
// two CTAs per SM.  (More channels stay on the cp.async-staged kernel, which
// measured faster there: 32 -> 32 on 1280 x 720, 795 us against 806-824 us
// for TMA configurations with 5 or 7 pixels per thread.)
#include "conv_tma.cuh"

namespace sc {

// <K, F_TB, W_T, TH, H_T, C_SH, NSTAGE, MINB, PAIRC>
// 16 or fewer output channels; cudaErrorNotSupported where the kernel does
// not apply (the caller then uses conv_general_k5.cu's configurations).
cudaError_t launch_conv_tma_k5_narrow(const ConvArgs &a, cudaStream_t st)
{
    if (a.Cout <= 4) return launch_conv_tma<TmaCfg<5, 4, 5, 4, 1, 8, 2, 2, false>>(a, st);
    if (a.Cout <= 8) return launch_conv_tma<TmaCfg<5, 8, 5, 4, 1, 8, 2, 2, false>>(a, st);
    return launch_conv_tma<TmaCfg<5, 16, 5, 4, 1, 8, 2, 2, false>>(a, st);
}

}  // namespace sc
