// Instantiations of the TMA-staged direct convolution (conv_tma.cuh) for
// 3 x 3 filters and 16 or fewer output channels, and the driver's
// tensor-map encoder they share.
#include <mutex>

#include "autotune.h"
#include "conv_tma.cuh"

namespace sc {

PFN_cuTensorMapEncodeTiled_v12000 conv_tma_encoder()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// <K, F_TB, W_T, TH, H_T, C_SH, NSTAGE, MINB, PAIRC>
cudaError_t k3_tma_f4_w5_h4_pc(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 4, 5, 4, 1, 8, 3, 2, true>>(a, st);
}
cudaError_t k3_tma_f4_w5_h4(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 4, 5, 4, 1, 8, 3, 2, false>>(a, st);
}
cudaError_t k3_tma_f4_w5_h8_pc(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 4, 5, 8, 1, 8, 3, 1, true>>(a, st);
}
cudaError_t k3_tma_f4_w3_h4_pc(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 4, 3, 4, 1, 8, 3, 3, true>>(a, st);
}
cudaError_t k3_tma_f4_w5_h8r2(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 4, 5, 8, 2, 8, 2, 2, false>>(a, st);
}
// one CTA a SM with 8 consumer warps: a tile 8 rows high shares its halo
// rows among more output rows (10 staged rows for 8, against 6 for 4)
cudaError_t k3_tma_f4_w5_h8(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 4, 5, 8, 1, 8, 3, 1, false>>(a, st);
}
cudaError_t k3_tma_f4_w5_h8_s4(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 4, 5, 8, 1, 8, 4, 1, false>>(a, st);
}
cudaError_t k3_tma_f8_w5_h4(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 8, 5, 4, 1, 8, 3, 2, false>>(a, st);
}
cudaError_t k3_tma_f16_w5_h4(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 16, 5, 4, 1, 8, 3, 2, false>>(a, st);
}
cudaError_t k3_tma_f16_w3_h4(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 16, 3, 4, 1, 8, 2, 2, false>>(a, st);
}
// small images (16 -> 16 on 128 x 128): more, smaller CTAs so every SM
// takes part; 8-channel groups or 2-row tiles
cudaError_t k3_tma_f16_w3_h2(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 16, 3, 2, 1, 8, 2, 4, false>>(a, st);
}
cudaError_t k3_tma_f8_w3_h4(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 8, 3, 4, 1, 8, 2, 4, false>>(a, st);
}
cudaError_t k3_tma_f8_w3_h2(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 8, 3, 2, 1, 8, 2, 4, false>>(a, st);
}
cudaError_t k3_tma_f32_w7_h8(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 32, 7, 8, 1, 8, 3, 1, false>>(a, st);
}
cudaError_t k3_tma_f32_w5_h8(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 32, 5, 8, 1, 8, 3, 1, false>>(a, st);
}
cudaError_t k3_tma_f64_w7_h8(const ConvArgs &a, cudaStream_t st)
{
    return launch_conv_tma<TmaCfg<3, 64, 7, 8, 1, 8, 3, 1, false>>(a, st);
}

// Default for more than 16 output channels: 64 per CTA above 32, else 32
// with the pixel run (5 or 7) that leaves fewer columns past the image edge.
cudaError_t launch_conv_tma_k3_wide(const ConvArgs &a, cudaStream_t st)
{
    if (a.Cout > 32) return k3_tma_f64_w7_h8(a, st);
    const int waste40 = (a.W + 39) / 40 * 40 - a.W, waste56 = (a.W + 55) / 56 * 56 - a.W;
    return waste56 < waste40 ? k3_tma_f32_w7_h8(a, st) : k3_tma_f32_w5_h8(a, st);
}

// The default configuration of the shape's class with one copy per CTA left
// un-issued and waits bounded by timeout_ns (sc_test_conv_wait_expiry).
cudaError_t launch_conv_tma_k3_test(const ConvArgs &a, int drop_copy, unsigned long long timeout_ns,
                                    cudaStream_t st)
{
    if (a.Cout <= 4) return launch_conv_tma<TmaCfg<3, 4, 5, 4, 1, 8, 3, 2, false>>(a, st, drop_copy, timeout_ns);
    if (a.Cout <= 8) return launch_conv_tma<TmaCfg<3, 8, 5, 4, 1, 8, 3, 2, false>>(a, st, drop_copy, timeout_ns);
    if (a.Cout <= 16) return launch_conv_tma<TmaCfg<3, 16, 5, 4, 1, 8, 3, 2, false>>(a, st, drop_copy, timeout_ns);
    if (a.Cout <= 32) return launch_conv_tma<TmaCfg<3, 32, 5, 8, 1, 8, 3, 1, false>>(a, st, drop_copy, timeout_ns);
    return launch_conv_tma<TmaCfg<3, 64, 7, 8, 1, 8, 3, 1, false>>(a, st, drop_copy, timeout_ns);
}

// Default for 16 or fewer output channels: the TMA-staged kernel, one
// output-channel group per CTA; cudaErrorNotSupported where it does not
// apply (the caller then uses conv_general_k3n.cu's configurations).
cudaError_t launch_conv_tma_k3_narrow(const ConvArgs &a, cudaStream_t st)
{
    if (a.Cout <= 4) {
        // 8 x 160 tiles with one CTA a SM (10 staged rows for 8 output
        // rows) where they give every SM at least two; 4 output channels
        // from 32 take the narrow-output kernel (32 -> 4 on 1280 x 720:
        // 51.9 -> 48.8 us)
        const long long tiles8 = (long long)((a.W + 159) / 160) * ((a.H + 7) / 8) * a.N;
        if (tiles8 >= 2LL * device_sm_count()) {
            if (a.Cout == 4) {
                const cudaError_t e = k3_n4_h8_s4(a, st);
                if (e != cudaErrorNotSupported) return e;
            }
            return k3_tma_f4_w5_h8_s4(a, st);
        }
        return k3_tma_f4_w5_h4(a, st);
    }
    if (a.Cout <= 8) return k3_tma_f8_w5_h4(a, st);
    // 9-16 channels: 80 x 4 pixel tiles; where those give fewer tiles than
    // the device has SMs, 48 x 4 tiles spread the work over more SMs
    // (16 -> 16 on 128 x 128: 12.9 -> 10.9 us a call)
    const long long tiles80 = (long long)((a.W + 79) / 80) * ((a.H + 3) / 4) * a.N;
    if (tiles80 < device_sm_count()) return k3_tma_f16_w3_h4(a, st);
    return k3_tma_f16_w5_h4(a, st);
}

}  // namespace sc
