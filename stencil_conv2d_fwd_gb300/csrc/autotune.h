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

}  // namespace sc
