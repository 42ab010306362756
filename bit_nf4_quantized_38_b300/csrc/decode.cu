// Decode-sized forward (M <= 16 tokens) of the frozen-NF4 linear with LoRA:
//   Y = X W_hat^T + s (X A) B
// At decode batch sizes the layer is bound by HBM traffic on the packed 4-bit
// weights (0.5 B/param + 1/64 B/param of block codes), so this is a streaming
// GEMV / skinny GEMM, not a tile GEMM.  Three kernels, each launched as a
// programmatic dependent of the previous one so their launches overlap:
//
//   k_decode_xa      XA = X A on one cluster of CTAs (a slice of K each,
//                    8-byte loads of A rows), reduced in fixed order through
//                    distributed shared memory.
//   k_decode_stream  The weight stream.  Row tile t (16 weight rows) x its K
//                    range is cut into P equal pieces; each warp owns exactly
//                    one (tile, piece), so every warp moves the same number of
//                    bytes.  Per 128-wide K unit a lane loads 8 packed bytes of
//                    row g and of row g+8 for each of the two 64-blocks (a
//                    3-4-unit-deep register ring keeps the loads in flight), looks
//                    every byte (two codes) up in a 256-entry table of bf16
//                    level pairs held once per lane in shared memory (so
//                    lookups never conflict on a bank), and issues warp MMAs
//                    m16n8k16 with weight rows as M and tokens as N into a fresh
//                    fp32 accumulator per block, which is then scaled by the
//                    block constant.  The warp's 16 x 16 partial goes to its
//                    own slot of the workspace.
//   k_decode_out     Per row tile: the P partials summed in piece order,
//                    plus s XA B, written as bf16 Y.
//
// Numerics: the block constant multiplies fp32 partial sums of x * bf16(q[c]),
// so the weight used is q[c] (rounded once to bf16) times the fp32 constant,
// not bf16(q[c] * constant) as in the dequantized matrix; the two differ by
// one bf16 rounding per weight, inside the path's stated tolerance.  Results
// are deterministic (fixed reduction orders, no atomics).
#include <algorithm>

#include "common.cuh"
#include "decode.cuh"

namespace ql {
namespace {

constexpr int XA_CLUSTER = 16;  // non-portable cluster size (B300 allows 16)
constexpr int XA_THREADS = 256;
constexpr int XA_KMAX = 1024;   // K rows per CTA staged at once
constexpr int ST_WARPS = 8;
constexpr int ST_THREADS = ST_WARPS * 32;

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint2 ldg_stream_v2(const void *p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t byte_of(uint32_t w, uint32_t sel) {  // sel = 0x4440 | byte index
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(w), "r"(sel));
  return r;
}

// ---------------------------------------------------------------------------- XA
// XA[m][j] = sum_k X[m][k] A[k][j] (m < M <= MM, j < r), fp32.  CTA c of the
// cluster sums K rows [c K/C, (c+1) K/C): thread (row group, 4-column chunk)
// takes every rows_per_pass-th row with an 8-byte load of A; X comes from
// shared memory.  Partials are added in fixed order: row groups inside the
// CTA, then CTAs by CTA 0 through distributed shared memory.
template <int MM>
__global__ void __launch_bounds__(XA_THREADS)
k_decode_xa(const uint16_t *__restrict__ X, int M, int64_t K, const uint16_t *__restrict__ A, int r,
            float *__restrict__ XA, uint16_t *__restrict__ XA_out) {
  griddep_launch();
  __shared__ float part[16 * 128];
  __shared__ __align__(16) uint16_t xs[MM * XA_KMAX];
  uint32_t crank, csize;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(csize));
  const int64_t kc0 = (int64_t)crank * K / csize, kc1 = (int64_t)(crank + 1) * K / csize;
  const int tid = threadIdx.x;
  const int chunks = r / 4;                    // 4 columns per thread
  const int rpp = XA_THREADS / chunks;         // row groups
  const int ch = tid % chunks, rg = tid / chunks;
  float acc[MM][4];
#pragma unroll
  for (int m = 0; m < MM; ++m)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[m][c] = 0.0f;
  for (int64_t c0 = kc0; c0 < kc1; c0 += XA_KMAX) {
    const int nk = (int)min((int64_t)XA_KMAX, kc1 - c0);
    __syncthreads();
    for (int i = tid; i < MM * nk; i += XA_THREADS) {
      const int m = i / nk, k = i - m * nk;
      xs[m * XA_KMAX + k] = m < M ? X[(int64_t)m * K + c0 + k] : (uint16_t)0;
    }
    __syncthreads();
#pragma unroll 4
    for (int k = rg; k < nk; k += rpp) {
      const uint2 av = __ldg(reinterpret_cast<const uint2 *>(A + (c0 + k) * r + ch * 4));
      const float a4[4] = {bf16lo_to_f32(av.x), bf16hi_to_f32(av.x), bf16lo_to_f32(av.y), bf16hi_to_f32(av.y)};
#pragma unroll
      for (int m = 0; m < MM; ++m) {
        const float xv = bf16lo_to_f32(xs[m * XA_KMAX + k]);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[m][c] = fmaf(xv, a4[c], acc[m][c]);
      }
    }
  }
  for (int i = tid; i < 16 * 128; i += XA_THREADS) part[i] = 0.0f;
  __syncthreads();
  for (int g = 0; g < rpp; ++g) {
    if (rg == g) {
#pragma unroll
      for (int m = 0; m < MM; ++m)
#pragma unroll
        for (int c = 0; c < 4; ++c) part[m * 128 + ch * 4 + c] += acc[m][c];
    }
    __syncthreads();
  }
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (crank == 0) {
    const uint32_t local = (uint32_t)__cvta_generic_to_shared(part);
    for (int i = tid; i < M * r; i += XA_THREADS) {
      const int m = i / r, j = i - m * r;
      float s = 0.0f;
      for (uint32_t c = 0; c < csize; ++c) {
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                     : "=r"(remote)
                     : "r"(local + (uint32_t)(m * 128 + j) * 4u), "r"(c));
        float v;
        asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
        s += v;
      }
      XA[i] = s;
      if (XA_out) XA_out[i] = (uint16_t)(pack_bf16x2(s, 0.0f) & 0xFFFFu);
    }
  }
  // keep every CTA's shared memory alive until CTA 0 has read it
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------- weight stream
struct StreamArgs {
  const uint16_t *X;
  int M;
  int64_t K;
  const uint8_t *packed;
  const int8_t *code;
  const float *step;
  const float *mean;
  const float *absmax;
  int dq;
  int64_t N;
  int64_t tiles;  // ceil(N / 16)
  int P;          // pieces per row tile (warps per row tile)
  float *part;    // [tiles][P][16 rows][16 tokens]
  float q[16];
};

template <int MT>  // token tiles of 8
__global__ void __launch_bounds__(ST_THREADS, 2)
k_decode_stream(const StreamArgs a) {
  constexpr int RING = MT == 1 ? 4 : 3;  // 128-wide K units in flight per warp
  griddep_launch();
  __shared__ __align__(16) uint32_t tab[256 * 32];  // byte -> (bf16 q[hi], bf16 q[lo]), one copy per lane
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    // element 2j (high nibble) goes to the low half: it is the lower k of the MMA pair
    const uint32_t v = pack_bf16x2(a.q[(tid >> 4) & 15], a.q[tid & 15]);
    uint4 *dst = reinterpret_cast<uint4 *>(&tab[tid * 32]);
#pragma unroll
    for (int c = 0; c < 8; ++c) dst[c] = make_uint4(v, v, v, v);
  }
  __syncthreads();

  const int64_t item = (int64_t)blockIdx.x * ST_WARPS + warp;
  if (item >= a.tiles * a.P) {
    griddep_wait();
    return;
  }
  const int64_t rt = item / a.P;
  const int piece = (int)(item - rt * a.P);
  const int64_t upt = (a.K + 127) >> 7, nb_row = a.K >> 6;
  const int64_t u0 = piece * upt / a.P, u1 = (piece + 1) * upt / a.P;
  const int g = lane >> 2, t = lane & 3;
  const int64_t rowg = rt * 16 + g, rowg8 = rowg + 8;
  const bool vg = rowg < a.N, vg8 = rowg8 < a.N;
  const int64_t ldw = a.K >> 1;
  const uint8_t *pg = a.packed + (vg ? rowg : 0) * ldw + t * 8;
  const uint8_t *pg8 = a.packed + (vg8 ? rowg8 : 0) * ldw + t * 8;
  const uint32_t tl = (uint32_t)__cvta_generic_to_shared(tab) + (uint32_t)lane * 4u;
  const float mu = a.dq ? __ldg(a.mean) : 0.0f;

  const uint16_t *xr[MT];
  bool xv[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int tok = mt * 8 + g;
    xv[mt] = tok < a.M;
    xr[mt] = a.X + (xv[mt] ? tok : 0) * a.K + t * 16;
  }

  float acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[mt][i] = 0.0f;

  // ring of in-flight units: packed bytes and raw block constants
  uint2 rw[RING][2][2];   // [slot][row g / g+8][block]
  float rm[RING][2][2];   // raw code as float (double quant) or absmax
  float rs[RING][2][2];   // DQ step per row and block (a block pair can straddle a 256-block group)
  auto issue = [&](int slot, int64_t u) {
    const int64_t kb0 = u * 2;
    const bool b1 = kb0 + 1 < nb_row;  // K % 128 == 64: the last unit has one block
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const bool v = h ? vg8 : vg;
      const int64_t row = h ? rowg8 : rowg;
      const uint8_t *p = h ? pg8 : pg;
      rw[slot][h][0] = v ? ldg_stream_v2(p + kb0 * 32) : make_uint2(0, 0);
      rw[slot][h][1] = (v && b1) ? ldg_stream_v2(p + (kb0 + 1) * 32) : make_uint2(0, 0);
      const int64_t b = row * nb_row + kb0;
      if (a.dq) {
        rm[slot][h][0] = v ? (float)__ldg(a.code + b) : 0.0f;
        rm[slot][h][1] = (v && b1) ? (float)__ldg(a.code + b + 1) : 0.0f;
        rs[slot][h][0] = v ? __ldg(a.step + (b >> 8)) : 0.0f;
        rs[slot][h][1] = (v && b1) ? __ldg(a.step + ((b + 1) >> 8)) : 0.0f;
      } else {
        rm[slot][h][0] = v ? __ldg(a.absmax + b) : 0.0f;
        rm[slot][h][1] = (v && b1) ? __ldg(a.absmax + b + 1) : 0.0f;
        rs[slot][h][0] = rs[slot][h][1] = 0.0f;
      }
    }
  };

#pragma unroll
  for (int s = 0; s < RING; ++s)
    if (u0 + s < u1) issue(s, u0 + s);

  for (int64_t ub = u0; ub < u1; ub += RING) {
#pragma unroll
    for (int s = 0; s < RING; ++s) {
      const int64_t u = ub + s;
      if (u >= u1) break;
      const int64_t kb0 = u * 2;
      const int nblk = (kb0 + 1 < nb_row) ? 2 : 1;
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        if (blk >= nblk) break;
        // block constants, decoded after their loads have landed
        float mh0 = rm[s][0][blk], mh1 = rm[s][1][blk];
        if (a.dq) {
          mh0 = __fadd_rn(__fmul_rn(mh0, rs[s][0][blk]), mu);
          mh1 = __fadd_rn(__fmul_rn(mh1, rs[s][1][blk]), mu);
        }
        uint4 xf[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint4 *src = reinterpret_cast<const uint4 *>(xr[mt] + (kb0 + blk) * 64);
          xf[mt][0] = xv[mt] ? __ldg(src) : make_uint4(0, 0, 0, 0);
          xf[mt][1] = xv[mt] ? __ldg(src + 1) : make_uint4(0, 0, 0, 0);
        }
        float D[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) D[mt][i] = 0.0f;
        const uint32_t wg[2] = {rw[s][0][blk].x, rw[s][0][blk].y};
        const uint32_t wg8[2] = {rw[s][1][blk].x, rw[s][1][blk].y};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // MMA j takes k = 16 t + 4 j + [0, 4) of this block: bytes 2j and 2j+1
          const uint32_t wa = wg[j >> 1], wb = wg8[j >> 1];
          const uint32_t s0 = 0x4440u | (uint32_t)((j & 1) * 2), s1 = s0 + 1;
          uint32_t a0, a1, a2, a3;
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(a0) : "r"(tl + byte_of(wa, s0) * 128u));
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(a2) : "r"(tl + byte_of(wa, s1) * 128u));
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(a1) : "r"(tl + byte_of(wb, s0) * 128u));
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(a3) : "r"(tl + byte_of(wb, s1) * 128u));
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t *xw = reinterpret_cast<const uint32_t *>(&xf[mt][0]);
            mma16816(D[mt], a0, a1, a2, a3, xw[2 * j], xw[2 * j + 1]);
          }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          acc[mt][0] = fmaf(D[mt][0], mh0, acc[mt][0]);
          acc[mt][1] = fmaf(D[mt][1], mh0, acc[mt][1]);
          acc[mt][2] = fmaf(D[mt][2], mh1, acc[mt][2]);
          acc[mt][3] = fmaf(D[mt][3], mh1, acc[mt][3]);
        }
      }
      if (u + RING < u1) issue(s, u + RING);
    }
  }

  // the warp's 16 rows x 16 tokens partial -> its slot
  float *dst = a.part + item * 256;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    *reinterpret_cast<float2 *>(dst + g * 16 + mt * 8 + 2 * t) = make_float2(acc[mt][0], acc[mt][1]);
    *reinterpret_cast<float2 *>(dst + (g + 8) * 16 + mt * 8 + 2 * t) = make_float2(acc[mt][2], acc[mt][3]);
  }
  if (MT == 1)  // tokens 8..15 unused: keep the slot defined
    *reinterpret_cast<float4 *>(dst + (lane >> 1) * 16 + 8 + (lane & 1) * 4) = make_float4(0, 0, 0, 0);
  // this grid's completion must also cover k_decode_xa for the next kernel
  griddep_wait();
}

// ---------------------------------------------------------------------------- output
// One CTA per row tile: thread (row, token) sums the P partials in piece
// order, adds s * sum_j XA[token][j] B[j][row] and writes bf16 Y.
__global__ void __launch_bounds__(256)
k_decode_out(const float *__restrict__ part, int P, int64_t N, int M, const float *__restrict__ XA,
             const uint16_t *__restrict__ B, int r, float scale, uint16_t *__restrict__ Y) {
  __shared__ float sxa[16 * 128];
  __shared__ float sb[128 * 16];
  griddep_wait();
  const int64_t rt = blockIdx.x;
  const int tid = threadIdx.x;
  const int64_t n0 = rt * 16;
  for (int i = tid; i < M * r; i += 256) sxa[(i / r) * 128 + (i % r)] = XA[i];
  for (int i = tid; i < r * 16; i += 256) {
    const int j = i >> 4, c = i & 15;
    sb[j * 16 + c] = n0 + c < N ? bf16lo_to_f32(B[(int64_t)j * N + n0 + c]) : 0.0f;
  }
  __syncthreads();
  const int row = tid >> 4, m = tid & 15;
  const int64_t n = n0 + row;
  if (m >= M || n >= N) return;
  float s = 0.0f;
  const float *p = part + rt * P * 256 + row * 16 + m;
  for (int z = 0; z < P; ++z) s += p[z * 256];
  float l = 0.0f;
  for (int j = 0; j < r; ++j) l = fmaf(sxa[m * 128 + j], sb[j * 16 + row], l);
  Y[(int64_t)m * N + n] = (uint16_t)(pack_bf16x2(fmaf(scale, l, s), 0.0f) & 0xFFFFu);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

int decode_splits(int64_t N, int64_t K) {
  // Pieces per 16-row tile: as many as fit one warp each on the GPU (148 SMs x
  // 16 resident warps), at most 16, and keeping >= 2 units of 128 per warp.
  const int64_t tiles = (N + 15) / 16, upt = (K + 127) / 128;
  int64_t P = (148 * 16) / tiles;
  P = std::min<int64_t>(P, std::max<int64_t>(1, upt / 2));
  P = std::min<int64_t>(P, 16);
  return (int)std::max<int64_t>(P, 1);
}

size_t decode_ws(int64_t N, int64_t K, int r) {
  (void)r;
  const size_t tiles = (size_t)((N + 15) / 16);
  return up256(16 * 128 * 4) + up256(tiles * (size_t)decode_splits(N, K) * 256 * 4);
}

int launch_decode(const DecodeProblem &p, cudaStream_t st) {
  char *ws = static_cast<char *>(p.ws);
  float *xa = reinterpret_cast<float *>(ws);
  float *part = reinterpret_cast<float *>(ws + up256(16 * 128 * 4));
  const int64_t tiles = (p.N + 15) / 16;
  const int P = decode_splits(p.N, p.K);

  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    for (auto fn : {k_decode_xa<1>, k_decode_xa<4>, k_decode_xa<16>}) {
      int rc0 = check_cuda(cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
                           "decode XA: cluster attribute");
      if (rc0) return rc0;
    }
    attr_done[dev] = true;
  }
  {
    cudaLaunchConfig_t cx{};
    cx.gridDim = dim3(XA_CLUSTER);
    cx.blockDim = dim3(XA_THREADS);
    cx.stream = st;
    cudaLaunchAttribute ax[1];
    ax[0].id = cudaLaunchAttributeClusterDimension;
    ax[0].val.clusterDim.x = XA_CLUSTER;
    ax[0].val.clusterDim.y = 1;
    ax[0].val.clusterDim.z = 1;
    cx.attrs = ax;
    cx.numAttrs = 1;
    auto fn = p.M <= 1 ? k_decode_xa<1> : p.M <= 4 ? k_decode_xa<4> : k_decode_xa<16>;
    cudaError_t ex = cudaLaunchKernelEx(&cx, fn, p.X, (int)p.M, p.K, p.A, p.r, xa, p.XA_out);
    count_launch();
    int rc = check_cuda(ex, "decode XA launch");
    if (rc) return rc;
  }
  StreamArgs a{};
  a.X = p.X; a.M = (int)p.M; a.K = p.K;
  a.packed = p.w.packed; a.code = p.w.code; a.step = p.w.step; a.mean = p.w.mean; a.absmax = p.w.absmax;
  a.dq = p.w.dq; a.N = p.N; a.tiles = tiles; a.P = P; a.part = part;
  const Codebook &cb = codebook();
  for (int i = 0; i < 16; ++i) a.q[i] = cb.q[i];
  const unsigned blocks = (unsigned)((tiles * P + ST_WARPS - 1) / ST_WARPS);
  cudaError_t e = p.M <= 8 ? launch_pdl(k_decode_stream<1>, dim3(blocks), dim3(ST_THREADS), st, a)
                           : launch_pdl(k_decode_stream<2>, dim3(blocks), dim3(ST_THREADS), st, a);
  count_launch();
  int rc = check_cuda(e, "decode stream launch");
  if (rc) return rc;
  e = launch_pdl(k_decode_out, dim3((unsigned)tiles), dim3(256), st, (const float *)part, P, p.N, (int)p.M,
                 (const float *)xa, p.B, p.r, p.scale, p.Y);
  count_launch();
  return check_cuda(e, "decode output launch");
}

}  // namespace ql
