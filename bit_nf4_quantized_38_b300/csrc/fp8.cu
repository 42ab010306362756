// Operand preparation for the E4M3 forward (the FP8 variant of the training
// GEMM; E4M3 = 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, largest
// finite 448), one launch, two kinds of CTA:
//   CTAs [0, M)      row m of X: E_m = the largest exponent with
//                    amax_m * 2^E_m <= 448 (0 for an all-zero row), and the
//                    codes e4m3(x * 2^E_m) (exact scaling, then round to
//                    nearest even, saturating)
//   CTAs [M, M + G)  the largest |m_hat| over the weight's blocks (atomic max
//                    into a word the caller cleared), from which the GEMM
//                    takes the weight's exponent E the same way
#include <algorithm>

#include "common.cuh"
#include "fp8.cuh"
#include "ptx.cuh"

namespace ql {
namespace {

constexpr int kWmaxCtas = 148 * 2;
// rows of up to kRowRegs x (threads) x 8 elements stay in registers between
// the two passes; rows of up to 6144 elements take 128-thread CTAs (more rows
// in flight per SM), longer ones 256
constexpr int kRowRegs = 6;

__device__ __forceinline__ float absmax8(const uint4 v) {
  const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
  float a = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) a = fmaxf(a, fmaxf(fabsf(bf16lo_to_f32(wd[j])), fabsf(bf16hi_to_f32(wd[j]))));
  return a;
}

__device__ __forceinline__ uint2 codes8(const uint4 v, float sc) {
  const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
  uint32_t b[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    b[2 * j] = e4m3_code(__fmul_rn(bf16lo_to_f32(wd[j]), sc));
    b[2 * j + 1] = e4m3_code(__fmul_rn(bf16hi_to_f32(wd[j]), sc));
  }
  return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24), b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
}

// The row's amax over the CTA (a: this thread's share) -> E_m (stored by
// thread 0) and the exact scale 2^E_m.
__device__ __forceinline__ float row_scale(float a, float *red, int warp, int lane, int *row_exp, int64_t row) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if (lane == 0) red[warp] = a;
  __syncthreads();
  float amax = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
  const int E = e4m3_weight_exponent(amax);
  if (threadIdx.x == 0) row_exp[row] = E;
  return __uint_as_float((uint32_t)(E + 127) << 23);
}

__global__ void __launch_bounds__(256, 4) k_prep_e4m3(const uint4 *__restrict__ X, int64_t M, int64_t K,
                                                   uint2 *__restrict__ codes, int *__restrict__ row_exp, NF4View w,
                                                   float *__restrict__ wmax) {
  __shared__ float red[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((int64_t)blockIdx.x >= M) {
    // ------------------------------------------------ weight: max |m_hat|
    const int64_t n_b = w.rows * w.cols / 64;
    const float mu = w.dq ? __ldg(w.mean) : 0.0f;
    float m = 0.0f;
    const int64_t stride = (int64_t)(gridDim.x - M) * blockDim.x;
    for (int64_t b = ((int64_t)blockIdx.x - M) * blockDim.x + threadIdx.x; b < n_b; b += stride) {
      const float mh = w.dq ? __fadd_rn(__fmul_rn(dq_code_value(__ldg(w.code + b), w.dqt), __ldg(w.step + (b >> 8))),
                                        mu)
                            : __ldg(w.absmax + b);
      m = fmaxf(m, fabsf(mh));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int i = 1; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
      atomicMax(reinterpret_cast<int *>(wmax), __float_as_int(m));  // non-negative: bit order = value order
    }
    return;
  }
  // ------------------------------------------------ row of X
  const int64_t row = blockIdx.x, n8 = K / 8;
  const uint4 *x = X + row * n8;
  uint2 *c = codes + row * n8;
  if (n8 <= (int64_t)kRowRegs * blockDim.x) {
    // the whole row in registers: one read of X
    uint4 v[kRowRegs];
    float a = 0.0f;
#pragma unroll
    for (int j = 0; j < kRowRegs; ++j) {
      const int64_t i = threadIdx.x + (int64_t)j * blockDim.x;
      v[j] = i < n8 ? __ldg(x + i) : make_uint4(0u, 0u, 0u, 0u);
      a = fmaxf(a, absmax8(v[j]));
    }
    const float sc = row_scale(a, red, warp, lane, row_exp, row);
#pragma unroll
    for (int j = 0; j < kRowRegs; ++j) {
      const int64_t i = threadIdx.x + (int64_t)j * blockDim.x;
      if (i < n8) c[i] = codes8(v[j], sc);
    }
    return;
  }
  float a = 0.0f;
  for (int64_t i = threadIdx.x; i < n8; i += blockDim.x) a = fmaxf(a, absmax8(__ldg(x + i)));
  const float sc = row_scale(a, red, warp, lane, row_exp, row);
  for (int64_t i = threadIdx.x; i < n8; i += blockDim.x) c[i] = codes8(__ldg(x + i), sc);  // again (mostly L2)
}

}  // namespace

cudaError_t launch_prep_e4m3(const uint16_t *X, int64_t M, int64_t K, const NF4View &w, uint8_t *codes, int *row_exp,
                             float *wmax, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(wmax, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  const int64_t n_b = w.rows * w.cols / 64;
  const int64_t g = std::max<int64_t>(1, std::min<int64_t>((n_b + 255) / 256, kWmaxCtas));
  const unsigned threads = K <= 6144 ? 128u : 256u;
  k_prep_e4m3<<<(unsigned)(M + g), threads, 0, st>>>(reinterpret_cast<const uint4 *>(X), M, K,
                                                     reinterpret_cast<uint2 *>(codes), row_exp, w, wmax);
  count_launch();
  return cudaGetLastError();
}

}  // namespace ql
