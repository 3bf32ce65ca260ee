// Further tile configurations of the general direct convolution for 3 x 3
// filters and more than 16 output channels, tried by the first-call
// autotuner (filters resident in shared memory only), and the candidate
// tables of every output-channel class.
#include "autotune.h"
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_k3(const ConvArgs &a, cudaStream_t st);
const TuneCand *k3_narrow_table(const ConvArgs &a, int *n);
// instantiated in conv_general_k3.cu: each kernel configuration is
// instantiated in exactly one translation unit
cudaError_t k3_wide_w7_f64(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_wide_w8_f64(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_wide_w7_f32(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_wide_w8_f32(const ConvArgs &a, cudaStream_t st);

// Filters resident in shared memory, else not a candidate.
template <int F_TB, int W_T, int TH, int TW, int C_SH, int MINB>
static cudaError_t cand(const ConvArgs &a, cudaStream_t st)
{
    const size_t cin_pad = (size_t)(a.Cin + C_SH - 1) / C_SH * C_SH;
    if (a.Cin % C_SH != 0 || cin_pad * 9 * F_TB * 4 > kResidentFilterBytes) return cudaErrorNotSupported;
    return launch_gen<GenCfg<3, F_TB, W_T, TH, TW, C_SH, true, MINB>>(a, st);
}

static const TuneCand k3_wide64[] = {
    {"heuristic", launch_conv_general_k3},
    {"F64 W7 8x28", k3_wide_w7_f64},
    {"F64 W8 8x32", k3_wide_w8_f64},
    {"F64 W8 4x32 2/SM", cand<64, 8, 4, 32, 16, 2>},
    {"F64 W7 4x28 2/SM", cand<64, 7, 4, 28, 16, 2>},
    {"TMA F64 W7 8x28", k3_tma_f64_w7_h8},
};
static const TuneCand k3_wide32[] = {
    {"heuristic", launch_conv_general_k3},
    {"F32 W7 8x56", k3_wide_w7_f32},
    {"F32 W8 8x64", k3_wide_w8_f32},
    {"F32 W8 4x64 2/SM", cand<32, 8, 4, 64, 16, 2>},
    {"F32 W4 8x32", cand<32, 4, 8, 32, 16, 1>},
    {"TMA F32 W7 8x56", k3_tma_f32_w7_h8},
    {"TMA F32 W5 8x40", k3_tma_f32_w5_h8},
};
static const TuneCand k3_only_heuristic[] = {{"heuristic", launch_conv_general_k3}};

int k3_candidates(const ConvArgs &a, const TuneCand **out)
{
    int n = 0;
    if (a.Cout <= 16) {
        *out = k3_narrow_table(a, &n);
        return n;
    }
    if (a.Cin % 16 != 0) {
        *out = k3_only_heuristic;
        return 1;
    }
    if (a.Cout > 32) {
        *out = k3_wide64;
        return (int)(sizeof(k3_wide64) / sizeof(k3_wide64[0]));
    }
    *out = k3_wide32;
    return (int)(sizeof(k3_wide32) / sizeof(k3_wide32[0]));
}
}  // namespace sc
