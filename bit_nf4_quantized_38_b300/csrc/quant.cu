// NF4 quantization, double quantization of the block constants, and
// dequantization (QLoRA abstract, innovations (a) and (b); news write-up,
// "4-bit NormalFloat" and "Double Quantization" items).
//
// All three kernels are HBM-bound streams over the weight:
//   quantize   reads 2 B/param (bf16), writes 0.5 B/param + 4 B/block absmax
//   double q.  reads 4 B/block, writes 1 B/block + 4 B per 256 blocks
//   dequantize reads 0.5 B/param + 1 B/block, writes 2 B/param
// Every load and store of a warp is a contiguous, fully used run (the
// quantizer: 2 lanes per block, 64 B of bf16 in and 16 B of nibbles out per
// lane; the dequantizer: 8 lanes per block, 4 B of nibbles in and 16 B of
// bf16 out per lane).
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

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
// 32 contiguous bytes (a whole sector) in one load; p 32-byte aligned.
__device__ __forceinline__ void ld_stream32(const uint4 *p, uint4 &a, uint4 &b) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
               : "l"(p));
}

// Quantizer layout: 2 lanes per 64-element block, 32 consecutive elements
// (64 bytes of bf16) each, so one warp step covers 16 consecutive blocks
// (2 KB of W) and every lane writes 16 bytes of nibbles.
constexpr int kQLanes = 2;
constexpr int kQBlocksPerStep = 32 / kQLanes;
constexpr int kQCells = 256;                            // table rows: every byte value is a valid index
constexpr size_t kQTableBytes = (size_t)kQCells * 32 * 8;  // one 8-byte entry per cell and lane
// fma(x, 32, 1.5 * 2^23 + 32) = 0x4B400000 + rne(32 x + 32) as a bit pattern for x in [-1, 1]
constexpr float kCellRound = 12582944.0f;

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// NF4 code of w in a block with absmax m (2^-60 <= m <= 2^60), without a
// division.  The coding cell comes from w * (32 / m) with an approximate
// reciprocal: the cell is either the one of the exact quotient or its
// neighbour across a boundary no threshold lies near (the host checks that
// every threshold keeps 2^-16 from every boundary), so either cell decides
// correctly.  The decision x = RN(w / m) >= u is taken exactly as the sign of
// (w - m u) + m delta (two FMAs): t' = u - delta is the point where RN
// switches to u, no quotient of two bf16 values equals it, and near it
// w - m u is exact.  The result equals the code of the IEEE quotient for
// every pair of bf16 values with |w| <= m in the range (checked exhaustively
// on the host, also with the reciprocal perturbed by two ulps either way).
// kOneFma: no bf16 quotient lies between t' and u for this codebook (the host
// checks every threshold), so the sign of w - m u alone decides.
template <bool kOneFma>
__device__ __forceinline__ uint32_t nf4_code_fast(float w, float m, float r32, uint32_t tbase, uint32_t lane8) {
  const uint32_t cu = __float_as_uint(__fmaf_rn(w, r32, kCellRound));
  uint2 t;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(t.x), "=r"(t.y) : "r"(tbase + prmt(cu, lane8, 0x5504u)));
  const float e = __fmaf_rn(-m, __uint_as_float(t.x), w);
  const float v = kOneFma ? e : __fmaf_rn(m, __uint_as_float(t.y), e);
  // lower code + 1 sits in the low five bits of t.y; minus 1 when v < 0
  return (t.y & 31u) + (uint32_t)((int32_t)__float_as_uint(v) >> 31);
}

// The same decision from the IEEE quotient (block constants outside [2^-60, 2^60]).
__device__ __forceinline__ uint32_t nf4_code_ieee(float w, float m, uint32_t tbase, uint32_t lane8) {
  const float x = __fdiv_rn(w, m);
  const uint32_t cu = __float_as_uint(__fmaf_rn(x, 32.0f, kCellRound));
  uint2 t;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(t.x), "=r"(t.y) : "r"(tbase + prmt(cu, lane8, 0x5504u)));
  return (t.y & 31u) - 1u + (x >= __uint_as_float(t.x) ? 1u : 0u);
}

// Eight codes (elements 2j in the high nibble of byte j) -> one word.
__device__ __forceinline__ uint32_t pack8(const uint32_t (&c)[8]) {
  uint32_t o = c[0] * 16u + c[1];
  o = (c[2] * 16u + c[3]) * 0x100u + o;
  o = (c[4] * 16u + c[5]) * 0x10000u + o;
  return (c[6] * 16u + c[7]) * 0x1000000u + o;
}

// kWide: W is 32-byte aligned, so a lane's bytes load as whole sectors.
template <bool kOneFma, bool kWide>
__global__ void __launch_bounds__(kThreads, 3)
k_quantize(const uint4 *__restrict__ W, int64_t n_blocks, Codebook cb, uint4 *__restrict__ packed,
           float *__restrict__ absmax, double *__restrict__ sum_acc) {
  // Coding table, one copy per lane so lookups never conflict on a bank:
  // cell c, lane l at byte c * 256 + l * 8 (threshold bits, rounding step |
  // lower code + 1).  The address is one byte permute of the cell index (the
  // low byte of the rounding-constant sum) and l * 8; all 256 byte values
  // are rows, so no input (a NaN element included) reads outside the table.
  // Rows past the last cell hold no threshold and code 7 + 1.
  extern __shared__ __align__(16) uint2 table[];
  __shared__ double red[kThreads / 32];
  for (int i = threadIdx.x; i < kQCells * 32; i += kThreads) {
    const int c = i >> 5;
    table[i] = c < kCells ? make_uint2(__float_as_uint(cb.cell_u[c]), cb.cell_d[c])
                          : make_uint2(0x7F800000u, 0x30800000u | 8u);
  }
  __syncthreads();
  // the second level (a programmatic dependent) waits for this grid's
  // completion before it reads anything: it may launch now
  ptx::griddep_launch();

  const int lane = threadIdx.x & 31;
  const int sub = lane & (kQLanes - 1);
  const uint32_t tbase = (uint32_t)__cvta_generic_to_shared(table);
  const uint32_t lane8 = (uint32_t)lane * 8u;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int64_t stride = nwarps * kQBlocksPerStep;
  double local = 0.0;

  // A lane's 64 bytes as two whole 32-byte sectors: a load of half a sector
  // (16 bytes) would fetch the sector from L2 twice when L1 is bypassed.
  auto load = [&](int64_t base, uint4 (&v)[4]) {
    const int64_t b = base + lane / kQLanes;
    if (b < n_blocks && kWide) {
      ld_stream32(W + b * 8 + sub * 4, v[0], v[1]);
      ld_stream32(W + b * 8 + sub * 4 + 2, v[2], v[3]);
    } else if (b < n_blocks) {
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = ld_stream(W + b * 8 + sub * 4 + k);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = make_uint4(0, 0, 0, 0);
    }
  };
  uint4 nxt[4];
  int64_t base = warp * kQBlocksPerStep;
  if (base < n_blocks) load(base, nxt);
  for (; base < n_blocks; base += stride) {
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = nxt[k];
    if (base + stride < n_blocks) load(base + stride, nxt);
    const int64_t b = base + lane / kQLanes;
    float w[32];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t words[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        w[8 * k + 2 * i] = bf16lo_to_f32(words[i]);
        w[8 * k + 2 * i + 1] = bf16hi_to_f32(words[i]);
      }
    }
    float m = 0.0f;
#pragma unroll
    for (int e = 0; e < 32; ++e) m = fmaxf(m, fabsf(w[e]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    if (b >= n_blocks) continue;
    if (sub == 0) {
      absmax[b] = m;
      local += (double)m;
    }
    uint32_t out[4] = {0x77777777u, 0x77777777u, 0x77777777u, 0x77777777u};  // all-zero block: zero level
    if (m >= 0x1p-60f && m <= 0x1p60f) {
      const float r32 = rcp_approx(m) * 32.0f;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t c[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) c[e] = nf4_code_fast<kOneFma>(w[8 * h + e], m, r32, tbase, lane8);
        out[h] = pack8(c);
      }
    } else if (m > 0.0f) {  // block constants outside [2^-60, 2^60]: IEEE division
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t c[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) c[e] = nf4_code_ieee(w[8 * h + e], m, tbase, lane8);
        out[h] = pack8(c);
      }
    }
    packed[b * kQLanes + sub] = make_uint4(out[0], out[1], out[2], out[3]);
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

// One warp per group of 256 block constants, lane l holding constants
// 8l .. 8l + 7: the group's largest |c - mu| is a shuffle reduction, so a warp
// takes one memory round trip per group and no block barrier.  Launched as a
// programmatic dependent of the first level: it waits for it before reading.
constexpr int kDqWarps = 8;
__global__ void __launch_bounds__(kDqWarps * 32)
k_double_quant(const float *__restrict__ absmax, int64_t n_b, int64_t total_blocks, const double *__restrict__ sum,
               int dq_type, int8_t *__restrict__ code, float *__restrict__ step, float *__restrict__ mean) {
  __shared__ float mu_s;
  ptx::griddep_wait();  // the sum and the constants are complete
  // mu once per CTA (an fp64 division is slow on this GPU)
  if (threadIdx.x == 0) mu_s = __double2float_rn(__ddiv_rn(*sum, (double)total_blocks));
  __syncthreads();
  const float mu = mu_s;
  const int lane = threadIdx.x & 31;
  const bool e4m3 = dq_type == QL_DQ_E4M3;
  const bool vec_in = (reinterpret_cast<uintptr_t>(absmax) & 15) == 0;
  const bool vec_out = (reinterpret_cast<uintptr_t>(code) & 7) == 0;
  const int64_t n_2 = (n_b + 255) / 256;
  const int64_t nw = (int64_t)gridDim.x * kDqWarps;
  for (int64_t g = (int64_t)blockIdx.x * kDqWarps + (threadIdx.x >> 5); g < n_2; g += nw) {
    const int64_t i0 = g * 256 + lane * 8;
    const bool whole = i0 + 8 <= n_b;
    float c[8];
    if (whole && vec_in) {
      const float4 v0 = __ldg(reinterpret_cast<const float4 *>(absmax + i0));
      const float4 v1 = __ldg(reinterpret_cast<const float4 *>(absmax + i0 + 4));
      c[0] = v0.x; c[1] = v0.y; c[2] = v0.z; c[3] = v0.w;
      c[4] = v1.x; c[5] = v1.y; c[6] = v1.z; c[7] = v1.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) c[e] = i0 + e < n_b ? __ldg(absmax + i0 + e) : mu;  // past the end: c - mu = 0
    }
    float a = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      c[e] = __fsub_rn(c[e], mu);
      a = fmaxf(a, fabsf(c[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float st = __fdiv_rn(a, e4m3 ? 448.0f : 127.0f);
    uint32_t k[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      k[e] = 0u;
      if (st != 0.0f) {
        const float x = __fdiv_rn(c[e], st);
        k[e] = e4m3 ? (uint32_t)e4m3_code(x) : (uint32_t)(uint8_t)(int8_t)(int)fminf(fmaxf(rintf(x), -127.0f), 127.0f);
      }
    }
    if (whole && vec_out) {
      *reinterpret_cast<uint2 *>(code + i0) = make_uint2(k[0] | (k[1] << 8) | (k[2] << 16) | (k[3] << 24),
                                                         k[4] | (k[5] << 8) | (k[6] << 16) | (k[7] << 24));
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (i0 + e < n_b) code[i0 + e] = (int8_t)(uint8_t)k[e];
    }
    if (lane == 0) step[g] = st;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *mean = mu;
}

template <bool kDQ>
__global__ void __launch_bounds__(kThreads)
k_dequantize(const uint32_t *__restrict__ packed, int64_t n_blocks, const int8_t *__restrict__ code, int dq_type,
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
        if (kDQ) mh[u] = __fadd_rn(__fmul_rn(dq_code_value(__ldg(code + b), dq_type), __ldg(step + (b >> 8))), mu);
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
  const int64_t per_cta = (int64_t)kQBlocksPerStep * (kThreads / 32);
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

cudaError_t launch_quantize(const uint16_t *W, int64_t rows, int64_t cols, int quant_type, uint8_t *packed,
                            float *absmax, double *sum_acc, cudaStream_t st) {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_done[dev]) {
    // the table is the only shared memory the kernel needs; streaming loads bypass L1
    for (auto fn : {k_quantize<true, true>, k_quantize<false, true>, k_quantize<true, false>,
                    k_quantize<false, false>}) {
      if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQTableBytes);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    }
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int64_t n_blocks = rows * cols / 64;
  const Codebook &cb = codebook(quant_type);
  const int grid = grid_for_q(n_blocks, 3);
  const bool wide = (reinterpret_cast<uintptr_t>(W) & 31) == 0;
  auto fn = cb.one_fma ? (wide ? k_quantize<true, true> : k_quantize<true, false>)
                       : (wide ? k_quantize<false, true> : k_quantize<false, false>);
  fn<<<grid, kThreads, kQTableBytes, st>>>(reinterpret_cast<const uint4 *>(W), n_blocks, cb,
                                           reinterpret_cast<uint4 *>(packed), absmax, sum_acc);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_double_quant(const float *absmax, int64_t n_b, int64_t total_blocks, int dq_bs, int dq_type,
                                const double *sum, int8_t *code, float *step, float *mean, cudaStream_t st) {
  (void)dq_bs;  // 256, checked by the caller
  const int64_t n_2 = (n_b + 255) / 256;
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((n_2 + kDqWarps - 1) / kDqWarps, (int64_t)sms * 8));
  // a programmatic dependent of the first-level kernel: its launch overlaps
  // that kernel's tail, and it waits for it before reading
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kDqWarps * 32);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_double_quant, absmax, n_b, total_blocks, sum, dq_type, code, step, mean);
  count_launch();
  return e;
}

cudaError_t launch_dequantize(const ql_nf4_tensor &q, uint16_t *W_out, cudaStream_t st) {
  const int64_t n_blocks = q.rows * q.cols / 64;
  const int g = grid_for(n_blocks, 8);
  const uint32_t *p = reinterpret_cast<const uint32_t *>(q.packed);
  uint4 *o = reinterpret_cast<uint4 *>(W_out);
  if (q.dq_blocksize)
    k_dequantize<true><<<g, kThreads, 0, st>>>(p, n_blocks, q.absmax_code, q.dq_type, q.dq_step, q.dq_mean,
                                               nullptr, codebook(q.quant_type), o);
  else
    k_dequantize<false><<<g, kThreads, 0, st>>>(p, n_blocks, nullptr, 0, nullptr, nullptr, q.absmax,
                                                codebook(q.quant_type), o);
  count_launch();
  return cudaGetLastError();
}

}  // namespace ql
