// Launch interface of the decode-sized forward (internal).
#pragma once
#include "tc_gemm.cuh"

namespace ql {

struct DecodeProblem {
  const uint16_t *X;  // M x K bf16, M <= 16
  int64_t M, K, N;
  NF4View w;          // N x K
  const uint16_t *A;  // K x r
  const uint16_t *B;  // r x N
  int r;
  float scale;
  uint16_t *Y;        // M x N
  uint16_t *XA_out;   // M x r or null
  void *ws;
};

size_t decode_ws(int64_t N, int64_t K, int r);
int launch_decode(const DecodeProblem &p, cudaStream_t st);

}  // namespace ql
