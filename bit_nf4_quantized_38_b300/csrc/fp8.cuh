// Operand preparation for the E4M3 forward (internal; see fp8.cu).
#pragma once
#include "common.cuh"
#include "tc_gemm.cuh"

namespace ql {

// codes [M][K] = e4m3(x * 2^E_m) per X row with row_exp[M] = E_m, and
// partial maxima of |m_hat| over the weight's blocks in wpart[0, *n_wpart)
// (at most kWmaxParts; max |m_hat| = the largest of them: wmax_of_warp).  K % 8
// == 0; X 16- and codes 8-byte aligned.  free_: X and the weight are not
// written, and codes, row_exp and wpart not read or written, by any kernel
// that may still be running (the kernel then runs alongside its predecessor).
// swapped: each pair of codes stored in swapped order (element 2j + 1 at byte
// 2j), the order of the forward GEMM's E4M3 weight rows along the reduction.
constexpr int kWmaxParts = 148;
cudaError_t launch_prep_e4m3(const uint16_t *X, int64_t M, int64_t K, const NF4View &w, uint8_t *codes, int *row_exp,
                             float *wpart, int *n_wpart, bool free_, bool swapped, cudaStream_t st);

// max |m_hat| from the partial maxima, by one warp (every lane gets it).
__device__ __forceinline__ float wmax_of_warp(const float *wpart, int n) {
  float m = 0.0f;
  for (int i = (int)(threadIdx.x & 31); i < n; i += 32) m = fmaxf(m, __ldg(wpart + i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

// 2^(-E_m - E): the factor of output row m (E from the weight's max |m_hat|).
__device__ __forceinline__ float e4m3_row_factor(int row_exp, float wmax) {
  const int t = -row_exp - e4m3_weight_exponent(wmax);
  return __uint_as_float((uint32_t)(t + 127) << 23);  // t in [-120, 120]
}

}  // namespace ql
