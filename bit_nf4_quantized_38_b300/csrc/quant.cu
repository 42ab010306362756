// NF4 quantization, double quantization of the block constants, and
// dequantization (QLoRA abstract, innovations (a) and (b); news write-up,
// "4-bit NormalFloat" and "Double Quantization" items).
//
// All three kernels are HBM-bound streams over the weight:
//   quantize   reads 2 B/param (bf16), writes 0.5 B/param + 4 B/block absmax
//   double q.  reads 4 B/block, writes 1 B/block + 4 B per 256 blocks
//   dequantize reads 0.5 B/param + 1 B/block, writes 2 B/param
// A warp covers 4 consecutive 64-element blocks per step (8 lanes per block,
// 16 B of bf16 or 4 B of nibbles per lane), so every load and store is a
// contiguous, fully used 128-512 B run.
#include "common.cuh"

namespace ql {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // warp steps in flight per thread

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// x = fl32(w / m) for |w| <= m, without a division per element: with
// r = RN(1/m) and x0 = RN(w r), the residual w - x0 m is exact under FMA and
// RN(x0 + residual * r) is the correctly rounded quotient (Markstein's
// correction step for division).  Checked exhaustively over every pair of
// bf16 values with |w| <= m and m in [2^-60, 2^60]: it equals the IEEE
// quotient whenever |x| >= 2^-12; smaller quotients (only with subnormal w)
// may differ in the last bit, but every quotient that small codes to the zero
// level either way.  Blocks with m outside that range take the IEEE division.
__device__ __forceinline__ float quotient(float w, float m, float r) {
  float x0 = __fmul_rn(w, r);
  float res = __fmaf_rn(-x0, m, w);
  return __fmaf_rn(res, r, x0);
}

// Quantizer layout: 4 lanes per 64-element block, 16 consecutive elements
// (32 bytes of bf16) each, so one warp step covers 8 consecutive blocks
// (1 KB of W) and writes 8 bytes of nibbles per lane.
constexpr int kQLanes = 4;
constexpr int kQBlocksPerStep = 32 / kQLanes;
constexpr int kQUnroll = 2;  // warp steps in flight per thread

// fma(x, 32, 1.5 * 2^23 + 32) has the bit pattern 0x4B400000 + rne(32 x + 32)
// for x in [-1, 1]; kCellTop is that of x = 1 (cell 64).  Finite x in [-1, 1]
// lie at or below it; NaN patterns (either sign) and anything above clamp to it.
constexpr uint32_t kCellTop = 0x4B400000u + 64u;
static_assert(kCells == 65, "cells 0..64");

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__global__ void __launch_bounds__(kThreads)
k_quantize(const uint4 *__restrict__ W, int64_t n_blocks, Codebook cb, uint2 *__restrict__ packed,
           float *__restrict__ absmax, double *__restrict__ sum_acc) {
  // Coding table, one copy per lane so lookups never conflict on a bank: cell
  // c, lane l at byte c * 256 + l * 8 (threshold bits, lower code).  The
  // lookup address comes from one byte permute of the cell index (the low
  // byte of the rounding-constant sum below) and l * 8.
  __shared__ __align__(16) uint2 table[kCells * 32];
  __shared__ double red[kThreads / 32];
  for (int i = threadIdx.x; i < kCells * 32; i += kThreads) {
    const int c = i >> 5;
    table[i] = make_uint2(__float_as_uint(cb.cell_u[c]), (uint32_t)cb.cell_lo[c]);
  }
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int sub = lane & (kQLanes - 1);
  const uint32_t tbase = (uint32_t)__cvta_generic_to_shared(table);
  const uint32_t lane8 = (uint32_t)lane * 8u;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  double local = 0.0;

  for (int64_t base = warp * kQBlocksPerStep * kQUnroll; base < n_blocks;
       base += nwarps * kQBlocksPerStep * kQUnroll) {
    uint4 v[kQUnroll][2];
#pragma unroll
    for (int u = 0; u < kQUnroll; ++u) {
      const int64_t b = base + u * kQBlocksPerStep + lane / kQLanes;
      const bool in = b < n_blocks;
      v[u][0] = in ? ld_stream(W + b * 8 + sub * 2) : make_uint4(0, 0, 0, 0);
      v[u][1] = in ? ld_stream(W + b * 8 + sub * 2 + 1) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kQUnroll; ++u) {
      const int64_t b = base + u * kQBlocksPerStep + lane / kQLanes;
      float w[16];
      const uint32_t words[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w,
                                 v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        w[2 * i] = bf16lo_to_f32(words[i]);
        w[2 * i + 1] = bf16hi_to_f32(words[i]);
      }
      float m = 0.0f;
#pragma unroll
      for (int e = 0; e < 16; ++e) m = fmaxf(m, fabsf(w[e]));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      if (b >= n_blocks) continue;
      if (sub == 0) {
        absmax[b] = m;
        local += (double)m;
      }
      uint32_t out[2] = {0x77777777u, 0x77777777u};  // all-zero block: the zero level everywhere
      if (m >= 0x1p-60f && m <= 0x1p60f) {
        const float r = __frcp_rn(m);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t code[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float x = quotient(w[8 * h + e], m, r);
            // rne(32 x + 32) in the low byte, through the 1.5 * 2^23 rounding constant;
            // the unsigned min keeps the cell index in [0, 64] for any input
            // (a NaN element gives cell 64 instead of reading past the table)
            const uint32_t cu = min(__float_as_uint(__fmaf_rn(x, 32.0f, 12582944.0f)), kCellTop);
            uint2 t;
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                         : "=r"(t.x), "=r"(t.y)
                         : "r"(tbase + prmt(cu, lane8, 0x5504u)));
            code[e] = t.y + (x >= __uint_as_float(t.x) ? 1u : 0u);
          }
          // element 2j -> high nibble of byte j: each byte as 16 hi + lo, the
          // bytes placed by multiply-adds (the fields never overlap)
          uint32_t o = code[0] * 16u + code[1];
          o = (code[2] * 16u + code[3]) * 0x100u + o;
          o = (code[4] * 16u + code[5]) * 0x10000u + o;
          o = (code[6] * 16u + code[7]) * 0x1000000u + o;
          out[h] = o;
        }
      } else if (m > 0.0f) {  // constants outside [2^-60, 2^60]: IEEE division
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t o = 0;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float x = __fdiv_rn(w[8 * h + e], m);
            const uint32_t cu = min(__float_as_uint(__fmaf_rn(x, 32.0f, 12582944.0f)), kCellTop);
            const uint2 t = table[((cu & 0xFFu) << 5) + lane];
            const uint32_t code = t.y + (x >= __uint_as_float(t.x) ? 1u : 0u);
            o |= code << (8 * (e >> 1) + ((e & 1) ? 0 : 4));
          }
          out[h] = o;
        }
      }
      packed[b * kQLanes + sub] = make_uint2(out[0], out[1]);
    }
  }

  // fp64 sum of this CTA's block absmax values (exact for real weights, so the
  // order of the atomics does not change the total)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
  if (lane == 0) red[threadIdx.x >> 5] = local;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int i = 0; i < kThreads / 32; ++i) s += red[i];
    if (s != 0.0) atomicAdd(sum_acc, s);
  }
}

__global__ void __launch_bounds__(256)
k_double_quant(const float *__restrict__ absmax, int64_t n_b, int64_t total_blocks, const double *__restrict__ sum,
               int8_t *__restrict__ code, float *__restrict__ step, float *__restrict__ mean) {
  __shared__ float red[8];
  const float mu = __double2float_rn(__ddiv_rn(*sum, (double)total_blocks));
  const int64_t g = blockIdx.x;
  const int64_t i = g * 256 + threadIdx.x;
  const bool valid = i < n_b;
  const float c = valid ? __fsub_rn(absmax[i], mu) : 0.0f;
  float a = fabsf(c);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  float a2 = red[0];
#pragma unroll
  for (int k = 1; k < 8; ++k) a2 = fmaxf(a2, red[k]);
  const float st = __fdiv_rn(a2, 127.0f);
  if (valid) {
    int k = 0;
    if (st != 0.0f) {
      float t = rintf(__fdiv_rn(c, st));
      t = fminf(fmaxf(t, -127.0f), 127.0f);
      k = (int)t;
    }
    code[i] = (int8_t)k;
  }
  if (threadIdx.x == 0) {
    step[g] = st;
    if (g == 0) *mean = mu;
  }
}

template <bool kDQ>
__global__ void __launch_bounds__(kThreads)
k_dequantize(const uint32_t *__restrict__ packed, int64_t n_blocks, const int8_t *__restrict__ code,
             const float *__restrict__ step, const float *__restrict__ mean,
             const float *__restrict__ absmax, Codebook cb, uint4 *__restrict__ out) {
  __shared__ float qtab[16 * 32];  // one copy of the levels per lane
  for (int i = threadIdx.x; i < 16 * 32; i += kThreads) qtab[i] = cb.q[i >> 5];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;
  const float *q = qtab + lane;
  const float mu = kDQ ? *mean : 0.0f;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  for (int64_t base = warp * 4 * kUnroll; base < n_blocks; base += nwarps * 4 * kUnroll) {
    uint32_t wd[kUnroll];
    float mh[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      int64_t b = base + u * 4 + (lane >> 3);
      wd[u] = 0;
      mh[u] = 0.0f;
      if (b < n_blocks) {
        wd[u] = __ldg(packed + b * 8 + sub);
        if (kDQ) mh[u] = __fadd_rn(__fmul_rn((float)__ldg(code + b), __ldg(step + (b >> 8))), mu);
        else mh[u] = __ldg(absmax + b);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      int64_t b = base + u * 4 + (lane >> 3);
      if (b >= n_blocks) continue;
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // byte j holds elements 2j (high) and 2j+1 (low)
        uint32_t byte = (wd[u] >> (8 * j)) & 0xFFu;
        float v0 = __fmul_rn(q[(byte >> 4) << 5], mh[u]);
        float v1 = __fmul_rn(q[(byte & 15u) << 5], mh[u]);
        o[j] = pack_bf16x2(v0, v1);
      }
      out[b * 8 + sub] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

int grid_for_q(int64_t n_blocks, int ctas_per_sm) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  const int64_t per_cta = (int64_t)kQBlocksPerStep * kQUnroll * (kThreads / 32);
  int64_t need = (n_blocks + per_cta - 1) / per_cta;
  int64_t g = (int64_t)sms * ctas_per_sm;
  if (need < g) g = need;
  return (int)(g < 1 ? 1 : g);
}

int grid_for(int64_t n_blocks, int ctas_per_sm) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  int64_t need = (n_blocks + 4 * kUnroll * (kThreads / 32) - 1) / (4 * kUnroll * (kThreads / 32));
  int64_t g = (int64_t)sms * ctas_per_sm;
  if (need < g) g = need;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_quantize(const uint16_t *W, int64_t rows, int64_t cols, uint8_t *packed,
                            float *absmax, double *sum_acc, cudaStream_t st) {
  const int64_t n_blocks = rows * cols / 64;
  k_quantize<<<grid_for_q(n_blocks, 8), kThreads, 0, st>>>(
      reinterpret_cast<const uint4 *>(W), n_blocks, codebook(), reinterpret_cast<uint2 *>(packed),
      absmax, sum_acc);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_double_quant(const float *absmax, int64_t n_b, int64_t total_blocks, int dq_bs,
                                const double *sum, int8_t *code, float *step, float *mean, cudaStream_t st) {
  (void)dq_bs;  // 256, checked by the caller
  const int64_t n_2 = (n_b + 255) / 256;
  k_double_quant<<<(unsigned)n_2, 256, 0, st>>>(absmax, n_b, total_blocks, sum, code, step, mean);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const ql_nf4_tensor &q, uint16_t *W_out, cudaStream_t st) {
  const int64_t n_blocks = q.rows * q.cols / 64;
  const int g = grid_for(n_blocks, 8);
  const uint32_t *p = reinterpret_cast<const uint32_t *>(q.packed);
  uint4 *o = reinterpret_cast<uint4 *>(W_out);
  if (q.dq_blocksize)
    k_dequantize<true><<<g, kThreads, 0, st>>>(p, n_blocks, q.absmax_code, q.dq_step, q.dq_mean,
                                               nullptr, codebook(), o);
  else
    k_dequantize<false><<<g, kThreads, 0, st>>>(p, n_blocks, nullptr, nullptr, nullptr, q.absmax,
                                                codebook(), o);
  count_launch();
  return cudaGetLastError();
}

}  // namespace ql
