// Operand preparation for the E4M3 forward (the FP8 variant of the training
// GEMM; E4M3 = 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, largest
// finite 448), one launch, two kinds of CTA:
//   CTAs [0, gw)      the largest |m_hat| over a share of the weight's blocks,
//                     one partial per CTA (wpart[c]; no atomics, nothing to
//                     clear): the consumers take the maximum of the gw
//                     partials and from it the weight's exponent E
//   CTAs [gw, grid)   rows of X in turn (a persistent grid): E_m = the largest
//                     exponent with amax_m * 2^E_m <= 448 (0 for an all-zero
//                     row), and the codes e4m3(x * 2^E_m) (exact scaling, then
//                     round to nearest even, saturating)
// A row CTA holds its row in registers and has the next row's loads in
// flight while it codes the current one (two register sets taking rows in
// turn), so every row costs one read of X and no exposed memory latency.
// Launched as a programmatic dependent of the previous kernel: with `free`
// it reads and writes nothing that kernel touches (the caller checks), so it
// runs alongside it and only its last CTA waits for it before exiting
// (completion still implies the predecessor's); otherwise it waits first.
#include <algorithm>

#include "common.cuh"
#include "fp8.cuh"
#include "ptx.cuh"

namespace ql {
namespace {


__device__ __forceinline__ float absmax8(const uint4 v) {
  const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
  float a = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) a = fmaxf(a, fmaxf(fabsf(bf16lo_to_f32(wd[j])), fabsf(bf16hi_to_f32(wd[j]))));
  return a;
}

// Eight codes e4m3(x 2^E_m) (the scaling is exact): the hardware conversion
// (round to nearest even, saturating at +-448), which equals e4m3_code for
// every finite input.  Element 2j in the low byte of pair j, or, with
// `swapped`, in the high byte (the pair order of the forward GEMM's weight
// rows).
__device__ __forceinline__ uint2 codes8(const uint4 v, float sc, bool swapped) {
  const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
  uint32_t h[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float lo = __fmul_rn(bf16lo_to_f32(wd[j]), sc), hi = __fmul_rn(bf16hi_to_f32(wd[j]), sc);
    h[j] = swapped ? ptx::cvt_e4m3x2(hi, lo) : ptx::cvt_e4m3x2(lo, hi);
  }
  return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}

// The row's amax over the CTA (a: this thread's share; red: this row's
// buffer of the two the CTA alternates, so one barrier per row suffices) ->
// E_m (stored by thread 0) and the exact scale 2^E_m.
__device__ __forceinline__ float row_scale(float a, float *red, int64_t row, int *row_exp) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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

// R: 16-byte pieces of a row per thread held in registers (rows of up to
// R x threads x 8 elements; longer rows are read twice).
template <int R>
__global__ void __launch_bounds__(R == 4 ? 128 : 256, R == 4 ? 8 : 3) k_prep_e4m3(const uint4 *__restrict__ X, int64_t M, int64_t K,
                                                                  uint2 *__restrict__ codes, int *__restrict__ row_exp,
                                                                  NF4View w, float *__restrict__ wpart, int gw,
                                                                  int free_, int swapped) {
  __shared__ float red[2][8];
  if (!free_) ptx::griddep_wait();
  ptx::griddep_launch();  // the dependents wait for this grid before reading its output
  // the CTA that waits for the predecessor at exit (free_); the grid's last
  // CTA is a row CTA
  const bool waiter = free_ && blockIdx.x == gridDim.x - 1 && threadIdx.x == 0;
  if ((int)blockIdx.x < gw) {
    // ------------------------------------------------ weight: max |m_hat|
    // 16 consecutive blocks per thread and load (one 16-byte load of codes,
    // or four of fp32 constants; the 16 share one second-level step), two
    // such loads in flight
    const int64_t n_b = w.rows * w.cols / 64, nch = (n_b + 15) / 16;
    const float mu = w.dq ? __ldg(w.mean) : 0.0f;
    const int64_t stride = (int64_t)gw * blockDim.x;
    float m = 0.0f;
    auto chunk = [&](int64_t c) {
      const int64_t b0 = c * 16;
      float v[16];
      if (b0 + 16 <= n_b) {
        if (w.dq) {
          const uint4 q = __ldg(reinterpret_cast<const uint4 *>(w.code + b0));
          const float st = __ldg(w.step + (b0 >> 8));
          const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int e = 0; e < 16; ++e)
            v[e] = __fadd_rn(__fmul_rn(dq_code_value((int8_t)(wd[e >> 2] >> (8 * (e & 3))), w.dqt), st), mu);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 f = __ldg(reinterpret_cast<const float4 *>(w.absmax + b0) + e);
            v[4 * e] = f.x; v[4 * e + 1] = f.y; v[4 * e + 2] = f.z; v[4 * e + 3] = f.w;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int64_t b = b0 + e;
          v[e] = 0.0f;
          if (b < n_b)
            v[e] = w.dq ? __fadd_rn(__fmul_rn(dq_code_value(__ldg(w.code + b), w.dqt), __ldg(w.step + (b >> 8))), mu)
                        : __ldg(w.absmax + b);
        }
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) m = fmaxf(m, fabsf(v[e]));
    };
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < nch; c += 2 * stride) {
      chunk(c);
      if (c + stride < nch) chunk(c + stride);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[0][threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int i = 1; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[0][i]);
      wpart[blockIdx.x] = m;
    }
    return;
  }
  // ------------------------------------------------ rows of X
  const int64_t n8 = K / 8, gr = (int64_t)gridDim.x - gw;
  const int nt = blockDim.x;
  int64_t row = (int64_t)blockIdx.x - gw;
  if (n8 <= (int64_t)R * nt) {
    auto load = [&](int64_t r, uint4 (&v)[R]) {
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int64_t i = threadIdx.x + (int64_t)j * nt;
        v[j] = (r < M && i < n8) ? __ldg(X + r * n8 + i) : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    auto code = [&](int64_t r, const uint4 (&v)[R], float *rd) {
      float a = 0.0f;
#pragma unroll
      for (int j = 0; j < R; ++j) a = fmaxf(a, absmax8(v[j]));
      const float sc = row_scale(a, rd, r, row_exp);
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int64_t i = threadIdx.x + (int64_t)j * nt;
        if (i < n8) codes[r * n8 + i] = codes8(v[j], sc, swapped != 0);
      }
    };
    uint4 va[R], vb[R];
    load(row, va);
#pragma unroll 1
    for (; row < M; row += 2 * gr) {
      load(row + gr, vb);
      code(row, va, red[0]);
      if (row + gr >= M) break;
      load(row + 2 * gr, va);
      code(row + gr, vb, red[1]);
    }
  } else {
    int par = 0;
#pragma unroll 1
    for (; row < M; row += gr, par ^= 1) {  // long rows: amax pass, then the row again (mostly from L2)
      const uint4 *x = X + row * n8;
      float a = 0.0f;
      for (int64_t i = threadIdx.x; i < n8; i += nt) a = fmaxf(a, absmax8(__ldg(x + i)));
      const float sc = row_scale(a, red[par], row, row_exp);
      for (int64_t i = threadIdx.x; i < n8; i += nt) codes[row * n8 + i] = codes8(__ldg(x + i), sc, swapped != 0);
    }
  }
  if (waiter) ptx::griddep_wait();  // this grid completes after its predecessor
}

template <int R>
int row_ctas_per_sm() {
  static int n[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!n[dev & 63]) {
    int k = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, k_prep_e4m3<R>, R == 4 ? 128 : 256, 0) != cudaSuccess ||
        k < 1)
      k = 1;
    n[dev & 63] = k;
  }
  return n[dev & 63];
}

int sm_count() {
  static int sms[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!sms[dev & 63]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    sms[dev & 63] = v > 0 ? v : 148;
  }
  return sms[dev & 63];
}

}  // namespace

cudaError_t launch_prep_e4m3(const uint16_t *X, int64_t M, int64_t K, const NF4View &w, uint8_t *codes, int *row_exp,
                             float *wpart, int *n_wpart, bool free_, bool swapped, cudaStream_t st) {
  const int64_t n_b = w.rows * w.cols / 64;
  const bool small = K <= 4 * 128 * 8;  // rows of up to 4096 elements: 128 threads x 4 pieces
  const int nt = small ? 128 : 256;
  const int64_t per_cta = (int64_t)nt * 16 * 2;  // blocks a weight CTA takes per round
  const int gw = (int)std::max<int64_t>(1, std::min<int64_t>((n_b + per_cta - 1) / per_cta, kWmaxParts));
  *n_wpart = gw;
  const int64_t per_sm = small ? row_ctas_per_sm<4>() : row_ctas_per_sm<6>();
  const int64_t gr = std::max<int64_t>(1, std::min<int64_t>(M, per_sm * sm_count()));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(gw + gr));
  cfg.blockDim = dim3((unsigned)nt);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint4 *x4 = reinterpret_cast<const uint4 *>(X);
  uint2 *c2 = reinterpret_cast<uint2 *>(codes);
  const int fr = free_ ? 1 : 0, sw = swapped ? 1 : 0;
  cudaError_t e = small ? cudaLaunchKernelEx(&cfg, k_prep_e4m3<4>, x4, M, K, c2, row_exp, w, wpart, gw, fr, sw)
                        : cudaLaunchKernelEx(&cfg, k_prep_e4m3<6>, x4, M, K, c2, row_exp, w, wpart, gw, fr, sw);
  count_launch();
  return e;
}

}  // namespace ql
