// Launch interface of the LoRA merge (internal).
#pragma once
#include "common.cuh"

namespace ql {

// W_out = bf16(w_hat + scale (A B)^T), W_out N x K bf16; arguments checked by the caller.
int launch_merge(const ql_nf4_tensor &W, const uint16_t *A, const uint16_t *B, int r, float scale, uint16_t *out,
                 cudaStream_t st);

}  // namespace ql
