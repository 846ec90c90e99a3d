// Tensor-core (tcgen05) path for bf16 activations: fused token-tile kernels.
#pragma once

#include "ttc_internal.h"

namespace ttc {

// True when the bf16 fused kernels handle this layer shape.
bool tc_supported(const LayerPlan& L);

// Bytes of workspace the fused path needs for its packed operands.
size_t tc_operand_bytes(const LayerPlan& L);

// y = ((x A) diag(D_d)) B with A (N x rd) and B (rd x M) the merged halves (f32,
// in the workspace); ws_off is the start of this path's operand region.
tt_status tc_forward(const LayerPlan& L, int64_t T, const void* x, const float* params,
                     const float* A, const float* B, void* y, void* ws, size_t ws_off,
                     cudaStream_t st);

// dx, dD_d (written to dDmid, honouring the prune convention and acc), and
// dA (N x rd), dB (rd x M) accumulated into the zeroed f32 buffers.
tt_status tc_backward(const LayerPlan& L, int64_t T, const void* x, const void* dy,
                      const float* params, const float* A, const float* B, void* dx,
                      float* dDmid, bool acc, float* dA, float* dB, void* ws, size_t ws_off,
                      cudaStream_t st);

}  // namespace ttc
