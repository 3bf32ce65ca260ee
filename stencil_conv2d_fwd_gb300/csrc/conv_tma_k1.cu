// Instantiations of the TMA-staged direct convolution (conv_tma.cuh) for
// 1 x 1 filters (no halo: a stage is the tile itself).
#include "conv_tma.cuh"

namespace sc {

// <K, F_TB, W_T, TH, H_T, C_SH, NSTAGE, MINB, PAIRC>
// 16 or fewer output channels; cudaErrorNotSupported where the kernel does
// not apply (the caller then uses conv_general_k1.cu's configurations).
cudaError_t launch_conv_tma_k1_narrow(const ConvArgs &a, cudaStream_t st)
{
    if (a.Cout <= 4) return launch_conv_tma<TmaCfg<1, 4, 5, 4, 1, 8, 3, 2, false>>(a, st);
    if (a.Cout <= 8) return launch_conv_tma<TmaCfg<1, 8, 5, 4, 1, 8, 3, 2, false>>(a, st);
    return launch_conv_tma<TmaCfg<1, 16, 5, 4, 1, 8, 3, 2, false>>(a, st);
}

// More than 16 output channels: 64 per CTA above 32, else 32.
cudaError_t launch_conv_tma_k1_wide(const ConvArgs &a, cudaStream_t st)
{
    if (a.Cout > 32) return launch_conv_tma<TmaCfg<1, 64, 7, 8, 1, 8, 3, 1, false>>(a, st);
    return launch_conv_tma<TmaCfg<1, 32, 5, 8, 1, 8, 3, 1, false>>(a, st);
}

}  // namespace sc
