// lm_head.cuh - internal interface between the fused LM-head kernel (lm_head.cu)
// and the acceptance entry point that finishes its rows (accept.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mars_lm_head {

// Vocabulary ranges (partials per row) the kernel uses for M rows and V entries.
int splits_for(int M, int V);

// Launches the fused head on `stream`: hidden [M, K] and weight [V, K] bf16 (K a
// multiple of 64), partials [M][nsplit] float4 = (max, argmax bits, sum of
// exp(x - max), -inf) over each vocabulary range.  Returns a MARS_* code.
int launch_partials(const uint16_t* hidden, const uint16_t* weight, int M, int K, int V, float4* partials,
                    int nsplit, int32_t* status, cudaStream_t stream);

}  // namespace mars_lm_head
