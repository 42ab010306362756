// LoRA merge for inference: W' = W_hat + s (A B)^T as a bf16 matrix (LoRA
// tutorial, Lit-LLaMA translation: after finetuning the low-rank update is
// added into the weight, W' = W + W_A W_B, so inference pays nothing for the
// adapter).  In row-major token form the update of weight row n, column k is
// s sum_j A[k][j] B[j][n].
//
// One pass over the frozen weight: a CTA owns a 64 x 128 tile of W'.  It
// stages the tile's packed nibbles and block constants, the 128 rows of A and
// the 64 columns of B it needs in shared memory; four warps compute the
// rank-r product with warp MMAs (m16n8k16, rows of W' as M, columns as N, the
// rank as K, zero-padded to 16), add it in fp32 to the dequantized weight
// w_hat = bf16(q[c] m_hat) of each element (one FMA: w_hat + s acc), round to
// bf16, and write the tile through shared memory with 16-byte stores.  HBM
// traffic is the weight's 0.5 + 1/64 bytes read and 2 bytes written per
// parameter (A and B are small and stay in L2).
#include <algorithm>

#include "common.cuh"
#include "merge.cuh"

namespace ql {
namespace {

constexpr int TM = 64;          // W' rows per CTA
constexpr int TK = 128;         // W' columns per CTA
constexpr int MTHREADS = 128;   // 4 warps x 16 rows
constexpr int OUT_LD = TK + 8;  // bf16 row stride of the output tile (bank spread)

struct MergeArgs {
  const uint8_t *packed;
  const int8_t *code;
  const float *step;
  const float *mean;
  const float *absmax;
  int dq;
  int dqt;  // second-level code (QL_DQ_INT8 or QL_DQ_E4M3)
  int N, K, r, rp;  // rp = r rounded up to 16
  const uint16_t *A;  // [K][r]
  const uint16_t *B;  // [r][N]
  float scale;
  uint16_t *out;      // [N][K]
  float q[16];
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared memory (bytes): A rows [TK][rp + 8], B rows [rp][TM + 8] (bf16, rows
// padded by 16 bytes so the 8 rows an ldmatrix reads fall in distinct banks),
// packed nibbles [TM][TK / 2], block constants [TM][TK / 64], levels [16],
// output tile [TM][OUT_LD] (bf16).
__host__ __device__ constexpr int a_ld(int rp) { return rp + 8; }
__host__ __device__ constexpr int b_ld() { return TM + 8; }
__host__ __device__ constexpr size_t merge_smem(int rp) {
  return (size_t)TK * a_ld(rp) * 2 + (size_t)rp * b_ld() * 2 + TM * (TK / 2) + TM * (TK / 64) * 4 + 16 * 4 +
         (size_t)TM * OUT_LD * 2;
}

__global__ void __launch_bounds__(MTHREADS) k_merge(const __grid_constant__ MergeArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int rp = a.rp;
  uint16_t *sA = reinterpret_cast<uint16_t *>(smem);
  uint16_t *sB = sA + TK * a_ld(rp);
  uint8_t *sP = reinterpret_cast<uint8_t *>(sB + rp * b_ld());
  float *sM = reinterpret_cast<float *>(sP + TM * (TK / 2));
  float *sQ = sM + TM * (TK / 64);
  uint16_t *sO = reinterpret_cast<uint16_t *>(sQ + 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int n0 = blockIdx.y * TM, k0 = blockIdx.x * TK;
  const int nrows = min(TM, a.N - n0);  // N % 8 == 0, so whole 8-row groups
  const int kcols = min(TK, a.K - k0);  // K % 64 == 0

  if (tid < 16) sQ[tid] = a.q[tid];
  // A rows k0 .. k0 + 127 (contiguous in global memory), zero past K and past r
  for (int i = tid; i < TK * (rp / 8); i += MTHREADS) {
    const int kr = i / (rp / 8), c8 = i % (rp / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (kr < kcols && c8 * 8 < a.r) v = __ldg(reinterpret_cast<const uint4 *>(a.A + (int64_t)(k0 + kr) * a.r) + c8);
    *reinterpret_cast<uint4 *>(sA + kr * a_ld(rp) + c8 * 8) = v;
  }
  // B columns n0 .. n0 + 63 of rows j < r, zero past N and past r
  for (int i = tid; i < rp * (TM / 8); i += MTHREADS) {
    const int j = i / (TM / 8), c8 = i % (TM / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (j < a.r && c8 * 8 < nrows) v = __ldg(reinterpret_cast<const uint4 *>(a.B + (int64_t)j * a.N + n0) + c8);
    *reinterpret_cast<uint4 *>(sB + j * b_ld() + c8 * 8) = v;
  }
  // packed nibbles of the tile (64 bytes per row) and its block constants
  for (int i = tid; i < TM * (TK / 32); i += MTHREADS) {
    const int nr = i / (TK / 32), c16 = i % (TK / 32);
    uint4 v = make_uint4(0x77777777u, 0x77777777u, 0x77777777u, 0x77777777u);
    if (nr < nrows && c16 * 32 < kcols)
      v = __ldg(reinterpret_cast<const uint4 *>(a.packed + (int64_t)(n0 + nr) * (a.K / 2) + k0 / 2) + c16);
    *reinterpret_cast<uint4 *>(sP + nr * (TK / 2) + c16 * 16) = v;
  }
  for (int i = tid; i < TM * (TK / 64); i += MTHREADS) {
    const int nr = i / (TK / 64), kb = i % (TK / 64);
    float m = 0.0f;
    if (nr < nrows && kb * 64 < kcols) {
      const int64_t b = (int64_t)(n0 + nr) * (a.K / 64) + k0 / 64 + kb;
      m = a.dq ? __fadd_rn(__fmul_rn(dq_code_value(__ldg(a.code + b), a.dqt), __ldg(a.step + (b >> 8))), __ldg(a.mean))
               : __ldg(a.absmax + b);
    }
    sM[i] = m;
  }
  __syncthreads();

  // warp w: W' rows 16 w .. 16 w + 15, all 128 columns (16 tiles of 8)
  float acc[TK / 8][4];
#pragma unroll
  for (int nt = 0; nt < TK / 8; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
  const uint32_t sA_u = (uint32_t)__cvta_generic_to_shared(sA), sB_u = (uint32_t)__cvta_generic_to_shared(sB);
  const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: which 8x8 matrix this lane addresses, and its row
  for (int kk = 0; kk < rp / 16; ++kk) {
    // A fragment (rows n, columns j) from B stored [j][n]: transposing loads of
    // the four 8 x 8 blocks (j 0-7 | 8-15) x (n 0-7 | 8-15)
    uint32_t a0, a1, a2, a3;
    {
      const int j = 16 * kk + (mi >> 1) * 8 + ri, n = 16 * warp + (mi & 1) * 8;
      ldsm_x4_t(sB_u + (uint32_t)((j * b_ld() + n) * 2), a0, a1, a2, a3);
    }
#pragma unroll
    for (int nt = 0; nt < TK / 8; nt += 2) {
      // B fragments (j x k) of tiles nt, nt + 1 from A stored [k][j]
      uint32_t b00, b01, b10, b11;
      const int k = nt * 8 + (mi >> 1) * 8 + ri, j = 16 * kk + (mi & 1) * 8;
      ldsm_x4(sA_u + (uint32_t)((k * a_ld(rp) + j) * 2), b00, b01, b10, b11);
      mma16816(acc[nt], a0, a1, a2, a3, b00, b01);
      mma16816(acc[nt + 1], a0, a1, a2, a3, b10, b11);
    }
  }

  // w_hat + s acc -> bf16 into the output tile
#pragma unroll
  for (int nt = 0; nt < TK / 8; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int nr = 16 * warp + g + 8 * h, kc = nt * 8 + 2 * t;  // kc even: one packed byte
      const uint32_t byte = sP[nr * (TK / 2) + kc / 2];
      const float m = sM[nr * (TK / 64) + kc / 64];
      const float w0 = bf16hi_to_f32(pack_bf16x2(0.0f, __fmul_rn(sQ[byte >> 4], m)));
      const float w1 = bf16hi_to_f32(pack_bf16x2(0.0f, __fmul_rn(sQ[byte & 15u], m)));
      const uint32_t o = pack_bf16x2(__fmaf_rn(a.scale, acc[nt][2 * h], w0), __fmaf_rn(a.scale, acc[nt][2 * h + 1], w1));
      *reinterpret_cast<uint32_t *>(sO + nr * OUT_LD + kc) = o;
    }
  __syncthreads();
  // 16-byte stores of the tile's valid part
  for (int i = tid; i < TM * (TK / 8); i += MTHREADS) {
    const int nr = i / (TK / 8), c8 = i % (TK / 8);
    if (nr < nrows && c8 * 8 < kcols)
      *reinterpret_cast<uint4 *>(a.out + (int64_t)(n0 + nr) * a.K + k0 + c8 * 8) =
          *reinterpret_cast<const uint4 *>(sO + nr * OUT_LD + c8 * 8);
  }
}

}  // namespace

int launch_merge(const ql_nf4_tensor &W, const uint16_t *A, const uint16_t *B, int r, float scale, uint16_t *out,
                 cudaStream_t st) {
  const int rp = std::max(16, (r + 15) / 16 * 16);
  const size_t smem = merge_smem(rp);
  static bool attr_done[64] = {};
  int dev = 0;
  int rc = check_cuda(cudaGetDevice(&dev), "qlora_merge: current device");
  if (rc) return rc;
  if (dev < 64 && !attr_done[dev]) {
    rc = check_cuda(cudaFuncSetAttribute(k_merge, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)merge_smem(128)),
                    "qlora_merge: shared-memory attribute");
    if (rc) return rc;
    attr_done[dev] = true;
  }
  MergeArgs a{};
  a.packed = W.packed; a.code = W.absmax_code; a.step = W.dq_step; a.mean = W.dq_mean; a.absmax = W.absmax;
  a.dq = W.dq_blocksize ? 1 : 0;
  a.dqt = W.dq_type;
  a.N = (int)W.rows; a.K = (int)W.cols; a.r = r; a.rp = rp;
  a.A = A; a.B = B; a.scale = scale; a.out = out;
  const Codebook &cb = codebook(W.quant_type);
  for (int i = 0; i < 16; ++i) a.q[i] = cb.q[i];
  dim3 grid((unsigned)((W.cols + TK - 1) / TK), (unsigned)((W.rows + TM - 1) / TM));
  k_merge<<<grid, MTHREADS, smem, st>>>(a);
  count_launch();
  return check_cuda(cudaGetLastError(), "qlora_merge launch");
}

}  // namespace ql
