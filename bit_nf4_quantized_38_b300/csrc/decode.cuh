// Launch interface of the decode-sized forward (internal).
#pragma once
#include "tc_gemm.cuh"

namespace ql {

struct DecodeProblem {
  const uint16_t *X;  // M x K bf16, M <= 32
  int64_t M, K, N;
  NF4View w;          // N x K
  const uint16_t *A;  // K x r
  const uint16_t *B;  // r x N
  int r;
  float scale;
  uint16_t *Y;        // M x N
  uint16_t *XA_out;   // M x r or null
  void *ws;           // any contents on entry; two halves, calls alternate
  int half;           // the half this call uses (the other one's call may still run)
  bool w_early;       // the previous grid writes none of the weight's arrays
  bool x_early;       // nor X, A or B
  bool ws_early;      // the previous grid touches none of this call's workspace half
};

size_t decode_ws(int64_t N, int64_t K, int r);
size_t decode_ws_half(int64_t N, int r);
// *early_dependents is set when the finishing kernel lets dependents launch
// before its own wait (the stream kernel then fills every SM).
int launch_decode(const DecodeProblem &p, cudaStream_t st, bool *early_dependents);

}  // namespace ql
