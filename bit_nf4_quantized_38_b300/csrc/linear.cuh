// Orchestration of the QLoRA linear forward and backward (internal).
#pragma once
#include "common.cuh"

namespace ql {

struct LinearArgs {
  const uint16_t *X, *dY, *A, *B, *XA_in;
  int64_t M;
  ql_nf4_tensor W;
  int32_t r;
  float scale;
  uint16_t *Y, *XA, *dX;
  float *dA, *dB;
  void *ws;
  size_t ws_bytes;
  cudaStream_t stream;
};

size_t linear_fwd_ws(int64_t M, int64_t N, int64_t K, int32_t r);
size_t linear_bwd_ws(int64_t M, int64_t N, int64_t K, int32_t r);
int linear_fwd(const LinearArgs &a);
int linear_bwd(const LinearArgs &a);
// The E4M3 forward (main product on E4M3 operands, LoRA term in bf16).
size_t linear_fwd_fp8_ws(int64_t M, int64_t N, int64_t K, int32_t r);
int linear_fwd_fp8(const LinearArgs &a);
// The E4M3 backward (dX main product on E4M3 operands; dA, dB as in bf16).
size_t linear_bwd_fp8_ws(int64_t M, int64_t N, int64_t K, int32_t r);
int linear_bwd_fp8(const LinearArgs &a);
// Record that a call other than a training linear was issued on `st` (its
// kernels do not let dependents start early; see linear.cu).
void note_other_call(cudaStream_t st);

}  // namespace ql
