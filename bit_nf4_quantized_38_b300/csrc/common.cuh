// Shared declarations of libqlora's CUDA sources (internal; the public ABI is
// include/qlora.h).
#pragma once
#include <cstring>

#include <cstdint>
#include <cstddef>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/qlora.h"

namespace ql {

// ---------------------------------------------------------------------------
// NF4 codebook, built on the host at load time from its definition (standard
// normal quantiles normalised to [-1, 1] with an exact zero) and handed to the
// kernels by value.

constexpr int kCells = 65;  // coding cells of width 1/32 over [-1, 1]

struct Codebook {
  float q[16];        // levels, ascending, fp32
  // Coding cells: an fp32 x in [-1, 1] falls in cell c = rne(32 x + 32).
  // Every cell holds at most one decision threshold; for x in cell c,
  // code(x) = cell_lo[c] + (x >= cell_u[c]).
  float cell_u[kCells];  // smallest fp32 above the cell's threshold (or +inf)
  int32_t cell_lo[kCells];
  // For the quantizer's division-free test: x = RN(w / m) >= u exactly when
  // w - m t' > 0, t' = (pred(u) + u) / 2 the rounding boundary below u (no
  // quotient of two bf16 values equals t').  t' = u - delta with delta a
  // power of two; cell_d holds delta's bits with cell_lo + 1 in its five low
  // mantissa bits (the perturbation, under 2^-18 delta, never changes the
  // sign of w - m u + m delta for bf16 w, m).  Cells without a threshold
  // hold delta = 2^-30.
  uint32_t cell_d[kCells];
  // True when no quotient w / m of two normal bf16 values lies in [t', u)
  // for any threshold: then w - m u >= 0 alone decides (one FMA, no delta).
  bool one_fma;
};

// Host: the code table of a quant type (QL_NF4 or QL_FP4; built once, thread-safe).
const Codebook &codebook(int quant_type = QL_NF4);

// ---------------------------------------------------------------------------
// errors

int set_error(int code, const char *fmt, ...);
int check_cuda(cudaError_t e, const char *what);

// Device status word set by bounded waits that give up (one per device).
enum : int { kStatusOk = 0, kStatusTimeout = 1 };
int *device_status_ptr();  // device address of the current device's word
void count_launch(int n = 1);  // kernels launched (process-wide counter)

// ---------------------------------------------------------------------------
// small device helpers

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Two fp32 -> packed bf16x2 with IEEE round-to-nearest-even; `lo` lands in the
// low 16 bits.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// E4M3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent
// 0 holds the subnormals m * 2^-9; largest finite 448 = 0x7E) from its
// definition.  Value of a code byte:
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 15u, m = code & 7u;
  const float v = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
  return (code & 0x80u) ? -v : v;
}
// Code of a finite fp32 x: round to nearest, ties to the even code,
// saturating at +-448 (the sign of x is kept, so -0 and negative values that
// round to 0 give 0x80).
__device__ __forceinline__ uint32_t e4m3_code(float x) {
  const uint32_t b = __float_as_uint(x), s = (b >> 24) & 0x80u;
  const float a = fabsf(x);
  if (!(a < 448.0f)) return s | 0x7Eu;
  if (a < 0.015625f) return s | (uint32_t)rintf(a * 512.0f);  // subnormal grid; 8 is 2^-6 (code 0x08)
  const uint32_t e = (b >> 23) & 0xFFu, mant = b & 0x7FFFFFu;
  uint32_t q = mant >> 20;
  const uint32_t rem = mant & 0xFFFFFu;
  if (rem > 0x80000u || (rem == 0x80000u && (q & 1u))) ++q;  // a carry into the exponent is right
  return s | (((e - 120u) << 3) + q);
}
// The weight's power-of-two scale for E4M3 main steps: the largest 2^E with
// maxm * 2^E <= 448 (maxm = f 2^e, f in [1, 2): E = 8 - e if f <= 1.75, else
// 7 - e), E clamped to [-60, 60]; 1 when maxm is 0.
__host__ __device__ __forceinline__ int e4m3_weight_exponent(float maxm) {
  if (!(maxm > 0.0f)) return 0;
  uint32_t b;
  memcpy(&b, &maxm, 4);
  const int e = (int)((b >> 23) & 0xFFu) - 127;
  uint32_t fb = (b & 0x7FFFFFu) | 0x3F800000u;
  float f;
  memcpy(&f, &fb, 4);
  int E = (f <= 1.75f ? 8 : 7) - e;
  return E < -60 ? -60 : (E > 60 ? 60 : E);
}
__device__ __forceinline__ float e4m3_weight_scale(float maxm) {
  return __uint_as_float((uint32_t)(e4m3_weight_exponent(maxm) + 127) << 23);
}

// Value of a second-level code byte (ql_nf4_tensor.dq_type).
__device__ __forceinline__ float dq_code_value(int8_t raw, int dq_type) {
  return dq_type == QL_DQ_E4M3 ? e4m3_value((uint8_t)raw) : (float)raw;
}

// ---------------------------------------------------------------------------
// launchers (quant.cu)

cudaError_t launch_quantize(const uint16_t *W, int64_t rows, int64_t cols, int quant_type, uint8_t *packed,
                            float *absmax, double *sum_acc, cudaStream_t st);
// mu = fl32(sum / total_blocks); codes and steps of the n_b blocks given.
cudaError_t launch_double_quant(const float *absmax, int64_t n_b, int64_t total_blocks, int dq_bs, int dq_type,
                                const double *sum, int8_t *code, float *step, float *mean, cudaStream_t st);
cudaError_t launch_dequantize(const ql_nf4_tensor &q, uint16_t *W_out, cudaStream_t st);

}  // namespace ql
