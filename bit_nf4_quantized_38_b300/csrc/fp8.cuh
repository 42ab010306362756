// Operand preparation for the E4M3 forward (internal; see fp8.cu).
#pragma once
#include "common.cuh"
#include "tc_gemm.cuh"

namespace ql {

// codes [M][K] = e4m3(x * 2^E_m) per X row with row_exp[M] = E_m, and
// *wmax = max |m_hat| of the weight (cleared here first).  K % 8 == 0; X 16-
// and codes 8-byte aligned.
cudaError_t launch_prep_e4m3(const uint16_t *X, int64_t M, int64_t K, const NF4View &w, uint8_t *codes, int *row_exp,
                             float *wmax, cudaStream_t st);

// 2^(-E_m - E): the factor of output row m (E from the weight's max |m_hat|).
__device__ __forceinline__ float e4m3_row_factor(int row_exp, float wmax) {
  const int t = -row_exp - e4m3_weight_exponent(wmax);
  return __uint_as_float((uint32_t)(t + 127) << 23);  // t in [-120, 120]
}

}  // namespace ql
