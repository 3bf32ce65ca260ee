// Further tile configurations of the general direct convolution for 3 x 3
// filters and 16 or fewer output channels, tried by the first-call
// autotuner (filters resident in shared memory only).
#include "autotune.h"
#include "conv_general.cuh"

namespace sc {
cudaError_t launch_conv_general_k3(const ConvArgs &a, cudaStream_t st);

template <int F_TB, int W_T, int TH, int TW, int MINB>
static cudaError_t cand_n(const ConvArgs &a, cudaStream_t st)
{
    const size_t cin_pad = (size_t)(a.Cin + 7) / 8 * 8;
    if (cin_pad * 9 * F_TB * 4 > kResidentFilterBytes) return cudaErrorNotSupported;
    return launch_gen<GenCfg<3, F_TB, W_T, TH, TW, 8, true, MINB>>(a, st);
}

static const TuneCand k3_n16[] = {
    {"heuristic", launch_conv_general_k3},
    {"F16 W8 4x128", cand_n<16, 8, 4, 128, 2>},
    {"F16 W4 8x64", cand_n<16, 4, 8, 64, 1>},
    {"TMA F16 W5 4x80", k3_tma_f16_w5_h4},
    {"TMA F16 W3 4x48", k3_tma_f16_w3_h4},
    {"TMA F16 W3 2x48", k3_tma_f16_w3_h2},
    {"TMA F8 W3 4x96", k3_tma_f8_w3_h4},
    {"TMA F8 W3 2x96", k3_tma_f8_w3_h2},
    {"small image 2x64", launch_conv_small},
};
static const TuneCand k3_n8[] = {
    {"heuristic", launch_conv_general_k3},
    {"F8 W8 4x256", cand_n<8, 8, 4, 256, 2>},
    {"TMA F8 W5 4x160", k3_tma_f8_w5_h4},
    {"small image 2x64", launch_conv_small},
};
static const TuneCand k3_n4[] = {
    {"heuristic", launch_conv_general_k3},
    {"F4 W8 4x256", cand_n<4, 8, 4, 256, 2>},
    {"F4 W4 2x128 4/SM", cand_n<4, 4, 2, 128, 4>},
    {"F4 W8 2x256 4/SM", cand_n<4, 8, 2, 256, 4>},
    {"TMA F4 W5 4x160 pc", k3_tma_f4_w5_h4_pc},
    {"TMA F4 W5 4x160", k3_tma_f4_w5_h4},
    {"TMA F4 W5 8x160 pc", k3_tma_f4_w5_h8_pc},
    {"TMA F4 W3 4x96 pc", k3_tma_f4_w3_h4_pc},
    {"TMA F4 W5 8x160 r2", k3_tma_f4_w5_h8r2},
    {"TMA F4 W5 8x160", k3_tma_f4_w5_h8},
    {"TMA F4 W5 8x160 4 stages", k3_tma_f4_w5_h8_s4},
    {"N4 W5 8x160 4 stages", k3_n4_h8_s4},
    {"N4 W5 8x160 c16", k3_n4_h8_c16},
    {"small image 2x64", launch_conv_small},
};

const TuneCand *k3_narrow_table(const ConvArgs &a, int *n)
{
    if (a.Cout > 8) {
        *n = (int)(sizeof(k3_n16) / sizeof(k3_n16[0]));
        return k3_n16;
    }
    if (a.Cout > 4) {
        *n = (int)(sizeof(k3_n8) / sizeof(k3_n8[0]));
        return k3_n8;
    }
    *n = (int)(sizeof(k3_n4) / sizeof(k3_n4[0]));
    return k3_n4;
}
}  // namespace sc
