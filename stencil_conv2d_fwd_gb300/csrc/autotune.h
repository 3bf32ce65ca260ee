// Tile-configuration candidates of the general direct convolution, for the
// first-call autotuner (autotune.cu).
#pragma once

#include "launch.h"

namespace sc {

struct TuneCand {
    const char *name;
    cudaError_t (*launch)(const ConvArgs &a, cudaStream_t st);   // cudaErrorNotSupported: not for this shape
};

// Candidates for 3 x 3 filters and Cin > 1: the heuristic dispatch first,
// then further tile configurations for the shape's output-channel class
// (conv_general_k3t.cu, conv_general_k3tn.cu).  Returns the count.
int k3_candidates(const ConvArgs &a, const TuneCand **out);

// TMA-staged configurations for 3 x 3 filters (conv_tma_k3.cu), named
// F<output channels per CTA>, W<pixels per thread>, <tile rows>, "r2": two
// tile rows per consumer warp; "pc": FMAs paired along input channels.
cudaError_t k3_tma_f4_w5_h4_pc(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f4_w5_h4(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f4_w5_h8_pc(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f4_w3_h4_pc(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f4_w5_h8r2(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f4_w5_h8(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f4_w5_h8_s4(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f8_w5_h4(const ConvArgs &a, cudaStream_t st);
// The narrow-output kernel (conv_narrow_k3.cu): 32 -> 4 channels, 8 x 160
// pixel tiles; "s4": four stages of 8 channels, "c16": two of 16.
cudaError_t k3_n4_h8_s4(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_n4_h8_c16(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f16_w5_h4(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f16_w3_h4(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f16_w3_h2(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f8_w3_h4(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f8_w3_h2(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f32_w7_h8(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f32_w5_h8(const ConvArgs &a, cudaStream_t st);
cudaError_t k3_tma_f64_w7_h8(const ConvArgs &a, cudaStream_t st);

}  // namespace sc
