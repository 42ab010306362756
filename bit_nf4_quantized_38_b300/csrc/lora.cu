// LoRA side products of the QLoRA linear (LoRA tutorial: dW = W_A W_B with
// rank r; QLoRA abstract: gradients flow into the adapters only):
//   XA = X A,  G = dY B^T,  dA = X^T (s G),  dB = s (XA)^T dY
// Each is a GEMM with a small side (r <= 128) and a long reduction, so the
// reduction is split across CTAs: every CTA writes an fp32 partial tile and a
// finalize kernel sums the partials in split order (deterministic), applies
// the scale and converts.  Tiles use the warp-level bf16 MMA (m16n8k16) fed by
// ldmatrix (.trans where the stored orientation needs it) from a cp.async
// double buffer.  These products are about 4% of the layer's flops.
#include "common.cuh"
#include "tc_gemm.cuh"

namespace ql {
namespace {

constexpr int SP = 64, SQ = 64, ST = 32;
constexpr int PAD = 8;
constexpr int SKINNY_THREADS = 128;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool kTrans>
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c, uint32_t &d) {
  if (kTrans)
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(addr));
  else
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared tile geometry (elements).  L: [ST][SP+PAD] when stored [t][p], else
// [SP][ST+PAD].  R: [SQ][ST+PAD] when stored [q][t], else [ST][SQ+PAD].
template <bool LTP>
struct LTile {
  static constexpr int rows = LTP ? ST : SP, ld = (LTP ? SP : ST) + PAD, elems = rows * ld;
};
template <bool RQT>
struct RTile {
  static constexpr int rows = RQT ? SQ : ST, ld = (RQT ? ST : SQ) + PAD, elems = rows * ld;
};

template <bool LTP, bool RQT>
__global__ void __launch_bounds__(SKINNY_THREADS)
k_skinny(const uint16_t *__restrict__ L, int64_t ldl, const uint16_t *__restrict__ R, int64_t ldr, int64_t P,
         int64_t Q, int64_t T, int64_t tps, float *__restrict__ part) {
  using LT = LTile<LTP>;
  using RT = RTile<RQT>;
  __shared__ __align__(16) uint16_t sL[2][LT::elems];
  __shared__ __align__(16) uint16_t sR[2][RT::elems];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t q0 = (int64_t)blockIdx.x * SQ, p0 = (int64_t)blockIdx.y * SP;
  const int64_t t_begin = (int64_t)blockIdx.z * tps;
  const int64_t t_end = min(T, t_begin + tps);
  float *out = part + (int64_t)blockIdx.z * P * Q;

  auto load = [&](int stage, int64_t t0) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = tid + h * SKINNY_THREADS;  // 256 16-byte chunks per tile
      {
        int row, col;
        const uint16_t *src;
        bool ok;
        if (LTP) {
          row = c >> 3; col = (c & 7) * 8;
          ok = (t0 + row < t_end) && (p0 + col < P);
          src = L + (ok ? (t0 + row) * ldl + p0 + col : 0);
        } else {
          row = c >> 2; col = (c & 3) * 8;
          ok = (p0 + row < P) && (t0 + col < t_end);
          src = L + (ok ? (p0 + row) * ldl + t0 + col : 0);
        }
        cp_async16((uint32_t)__cvta_generic_to_shared(&sL[stage][row * LT::ld + col]), src, ok);
      }
      {
        int row, col;
        const uint16_t *src;
        bool ok;
        if (RQT) {
          row = c >> 2; col = (c & 3) * 8;
          ok = (q0 + row < Q) && (t0 + col < t_end);
          src = R + (ok ? (q0 + row) * ldr + t0 + col : 0);
        } else {
          row = c >> 3; col = (c & 7) * 8;
          ok = (t0 + row < t_end) && (q0 + col < Q);
          src = R + (ok ? (t0 + row) * ldr + q0 + col : 0);
        }
        cp_async16((uint32_t)__cvta_generic_to_shared(&sR[stage][row * RT::ld + col]), src, ok);
      }
    }
    cp_async_commit();
  };

  float acc[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[i][j][k] = 0.0f;

  const int wp = (warp & 1) * 32, wq = (warp >> 1) * 32;
  const int nsteps = (int)((t_end - t_begin + ST - 1) / ST);
  if (nsteps > 0) load(0, t_begin);
  for (int it = 0; it < nsteps; ++it) {
    const int stage = it & 1;
    if (it + 1 < nsteps) {
      load(stage ^ 1, t_begin + (int64_t)(it + 1) * ST);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < ST; kk += 16) {
      uint32_t a[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int mi = lane >> 3, r8 = lane & 7;
        int row, col;
        if (LTP) {  // stored [t][p]: matrices (t,p) offsets (0,0) (0,8) (8,0) (8,8)
          row = kk + (mi >> 1) * 8 + r8;
          col = wp + i * 16 + (mi & 1) * 8;
        } else {    // stored [p][t]
          row = wp + i * 16 + (lane & 15);
          col = kk + (lane >> 4) * 8;
        }
        ldsm_x4<LTP>((uint32_t)__cvta_generic_to_shared(&sL[stage][row * LT::ld + col]), a[i][0], a[i][1],
                     a[i][2], a[i][3]);
      }
      uint32_t b[4][2];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int mi = lane >> 3, r8 = lane & 7;
        int row, col;
        if (RQT) {  // stored [q][t]: matrices (q,t) offsets (0,0) (0,8) (8,0) (8,8)
          row = wq + jj * 16 + (mi >> 1) * 8 + r8;
          col = kk + (mi & 1) * 8;
        } else {    // stored [t][q]: matrices (t,q) offsets (0,0) (8,0) (0,8) (8,8)
          row = kk + (mi & 1) * 8 + r8;
          col = wq + jj * 16 + (mi >> 1) * 8;
        }
        ldsm_x4<!RQT>((uint32_t)__cvta_generic_to_shared(&sR[stage][row * RT::ld + col]), b[2 * jj][0],
                      b[2 * jj][1], b[2 * jj + 1][0], b[2 * jj + 1][1]);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma16816(acc[i][j], a[i], b[j][0], b[j][1]);
    }
    __syncthreads();
  }

  const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int64_t p = p0 + wp + i * 16 + g + hh * 8;
        const int64_t q = q0 + wq + j * 8 + 2 * t4;
        if (p < P && q < Q)
          *reinterpret_cast<float2 *>(out + p * Q + q) = make_float2(acc[i][j][2 * hh], acc[i][j][2 * hh + 1]);
      }
}

__global__ void k_finalize_bf16(const float *__restrict__ part, int splits, int64_t P, int64_t Q, float scale,
                                uint16_t *__restrict__ out_pad, int qp, uint16_t *__restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= P * qp) return;
  const int64_t p = i / qp, q = i % qp;
  uint16_t v = 0;
  if (q < Q) {
    float s = 0.0f;
    for (int z = 0; z < splits; ++z) s += part[(int64_t)z * P * Q + p * Q + q];
    v = (uint16_t)(pack_bf16x2(__fmul_rn(s, scale), 0.0f) & 0xFFFFu);
    if (out) out[p * Q + q] = v;
  }
  out_pad[i] = v;
}

__global__ void k_finalize_f32(const float *__restrict__ part, int splits, int64_t n, float scale,
                               float *__restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float s = 0.0f;
  for (int z = 0; z < splits; ++z) s += part[(int64_t)z * n + i];
  out[i] = __fmul_rn(s, scale);
}

__global__ void k_pack_transpose(const uint16_t *__restrict__ B, int r, int64_t N, float scale,
                                 uint16_t *__restrict__ Bt, int rp) {
  __shared__ float tile[32][33];
  const int64_t n0 = (int64_t)blockIdx.x * 32;
  const int j0 = blockIdx.y * 32;
  for (int y = threadIdx.y; y < 32; y += blockDim.y) {  // read B[j][n], coalesced along n
    const int j = j0 + y;
    const int64_t n = n0 + threadIdx.x;
    tile[y][threadIdx.x] = (j < r && n < N) ? bf16lo_to_f32(B[(int64_t)j * N + n]) : 0.0f;
  }
  __syncthreads();
  for (int y = threadIdx.y; y < 32; y += blockDim.y) {  // write Bt[n][j], coalesced along j
    const int64_t n = n0 + y;
    const int j = j0 + threadIdx.x;
    if (n < N && j < rp)
      Bt[n * rp + j] = (uint16_t)(pack_bf16x2(__fmul_rn(tile[threadIdx.x][y], scale), 0.0f) & 0xFFFFu);
  }
}

__global__ void k_pack_pad(const uint16_t *__restrict__ A, int64_t K, int r, uint16_t *__restrict__ Ap, int rp) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= K * rp) return;
  const int64_t k = i / rp;
  const int j = (int)(i % rp);
  Ap[i] = j < r ? A[k * r + j] : (uint16_t)0;
}

unsigned blocks_for(int64_t n, int threads) { return (unsigned)((n + threads - 1) / threads); }

}  // namespace

int skinny_splits(int64_t P, int64_t Q, int64_t T) {
  const int64_t tiles = ((P + SP - 1) / SP) * ((Q + SQ - 1) / SQ);
  int64_t s = (2 * 148 + tiles - 1) / tiles;
  const int64_t max_s = std::max<int64_t>(1, T / 256);
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  return (int)s;
}

int launch_skinny(const SkinnyProblem &s, cudaStream_t st) {
  int64_t tps = (s.T + s.splits - 1) / s.splits;
  tps = (tps + ST - 1) / ST * ST;
  dim3 grid((unsigned)((s.Q + SQ - 1) / SQ), (unsigned)((s.P + SP - 1) / SP), (unsigned)s.splits);
  if (!s.l_tp && !s.r_qt)
    k_skinny<false, false><<<grid, SKINNY_THREADS, 0, st>>>(s.L, s.ldl, s.R, s.ldr, s.P, s.Q, s.T, tps, s.part);
  else if (!s.l_tp && s.r_qt)
    k_skinny<false, true><<<grid, SKINNY_THREADS, 0, st>>>(s.L, s.ldl, s.R, s.ldr, s.P, s.Q, s.T, tps, s.part);
  else if (s.l_tp && !s.r_qt)
    k_skinny<true, false><<<grid, SKINNY_THREADS, 0, st>>>(s.L, s.ldl, s.R, s.ldr, s.P, s.Q, s.T, tps, s.part);
  else
    k_skinny<true, true><<<grid, SKINNY_THREADS, 0, st>>>(s.L, s.ldl, s.R, s.ldr, s.P, s.Q, s.T, tps, s.part);
  count_launch();
  return check_cuda(cudaGetLastError(), "LoRA side GEMM launch");
}

int launch_finalize_bf16(const float *part, int splits, int64_t P, int64_t Q, float scale, uint16_t *out_pad,
                         int qp, uint16_t *out, cudaStream_t st) {
  k_finalize_bf16<<<blocks_for(P * qp, 256), 256, 0, st>>>(part, splits, P, Q, scale, out_pad, qp, out);
  count_launch();
  return check_cuda(cudaGetLastError(), "LoRA finalize launch");
}

int launch_finalize_f32(const float *part, int splits, int64_t P, int64_t Q, float scale, float *out,
                        cudaStream_t st) {
  k_finalize_f32<<<blocks_for(P * Q, 256), 256, 0, st>>>(part, splits, P * Q, scale, out);
  count_launch();
  return check_cuda(cudaGetLastError(), "LoRA finalize launch");
}

int launch_pack_transpose(const uint16_t *B, int r, int64_t N, float scale, uint16_t *Bt, int rp,
                          cudaStream_t st) {
  dim3 grid((unsigned)((N + 31) / 32), (unsigned)((rp + 31) / 32));
  k_pack_transpose<<<grid, dim3(32, 8), 0, st>>>(B, r, N, scale, Bt, rp);
  count_launch();
  return check_cuda(cudaGetLastError(), "LoRA pack launch");
}

int launch_pack_pad(const uint16_t *A, int64_t K, int r, uint16_t *Ap, int rp, cudaStream_t st) {
  k_pack_pad<<<blocks_for(K * rp, 256), 256, 0, st>>>(A, K, r, Ap, rp);
  count_launch();
  return check_cuda(cudaGetLastError(), "LoRA pack launch");
}

}  // namespace ql
