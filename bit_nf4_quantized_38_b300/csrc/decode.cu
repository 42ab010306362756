// Decode-sized forward (M <= 16 tokens) of the frozen-NF4 linear with LoRA:
//   Y = X W_hat^T + s (X A) B
// At decode batch sizes the layer is bound by HBM traffic on the packed 4-bit
// weights (0.5 B/param + 1/64 B/param of block codes), so this is a streaming
// GEMV / skinny GEMM, not a tile GEMM.  Two kernels; the second is launched as
// a programmatic dependent of the first, so it streams the weights while the
// first runs:
//
//   k_decode_xa      XA = X A on one cluster of CTAs, by warp MMAs: each CTA
//                    stages chunks of its K slice of A and X in shared memory
//                    (A swizzled so that transposing fragment loads never
//                    conflict), its warps split the chunk's k steps, and the
//                    warp and CTA partials are added in fixed order, the CTAs'
//                    through distributed shared memory.  It also clears the
//                    row-tile counters of the second kernel.
//   k_decode_stream  The weight stream.  Row tile t (16 weight rows) x K is
//                    cut into P pieces of whole 256-wide K boxes; each warp
//                    owns one (tile, piece) and a private 4-slot shared-memory
//                    ring that TMA fills with 16 x 128 B boxes of packed
//                    nibbles (128-byte swizzle, so the lanes' 8-byte reads
//                    spread over the banks).  Block constants are loaded three
//                    boxes ahead and X one 64-block ahead, so a warp waits on
//                    memory only when the ring itself runs dry.  Every byte
//                    (two codes) is looked up in a 256-entry table of bf16
//                    level pairs kept once per lane in shared memory (lookups
//                    never conflict on a bank); warp MMAs m16n8k16 with weight
//                    rows as M and tokens as N accumulate each 64-block in a
//                    fresh fp32 tile that is then scaled by the block constant.
//                    The warp's 16 x 16 partial goes to its own workspace
//                    slot; the last warp of a row tile to finish (counter per
//                    tile) adds the P partials in piece order, waits for XA,
//                    adds s XA B (warp MMAs) and writes Y.
//
// Numerics: the block constant multiplies fp32 partial sums of x * bf16(q[c]),
// so the weight used is q[c] (rounded once to bf16) times the fp32 constant,
// not bf16(q[c] * constant) as in the dequantized matrix; the two differ by
// one bf16 rounding per weight, inside the path's stated tolerance.  XA enters
// the LoRA product as a bf16 high part plus a bf16 low part (about 16
// significant bits).  Results are deterministic (fixed reduction orders).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "decode.cuh"
#include "ptx.cuh"

namespace ql {
namespace {

constexpr int XA_CLUSTER = 16;  // non-portable cluster size (B300 allows 16)
constexpr int XA_THREADS = 256;
constexpr int XA_WARPS = XA_THREADS / 32;
constexpr int XA_SMEM_MAX = 120 * 1024;  // leaves room for one weight-stream CTA on the SM
constexpr int ST_WARPS = 8;
constexpr int ST_THREADS = ST_WARPS * 32;
constexpr int RING = 4;          // boxes in flight per warp
constexpr int PD = 3;            // boxes of block constants loaded ahead
constexpr int BOX_K = 256;       // K values per box (128 bytes of nibbles per row)
constexpr int BOX_BYTES = 16 * 128;
constexpr size_t ST_SMEM = 1024 + (size_t)ST_WARPS * RING * BOX_BYTES + 256 * 32 * 4 + 1024;

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t byte_of(uint32_t w, uint32_t sel) {  // sel = 0x4440 | byte index
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(w), "r"(sel));
  return r;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Wait for phase `parity` of a barrier for at most `limit_ns`, ignoring any
// abort flag: used to let copies already in flight land before a warp that
// gave up exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = 100000000ull) {
  const uint64_t t0 = ptx::globaltimer();
#pragma unroll 1
  while (!ptx::mbar_try_wait(bar, parity) && ptx::globaltimer() - t0 < limit_ns) {
  }
}

// ---------------------------------------------------------------------------- XA
// Shared-memory position (in 16-byte units) of unit c (8 values of A[k][8c..])
// of row k of a staged A chunk with NT units per row.  Rows of 8 or more units
// XOR the unit with k mod 8; shorter rows XOR bits 0-2 of the linear unit
// index with bits 3-5.  Either way the 8 rows one transposing 8 x 8 fragment
// load touches land in 8 distinct bank groups.
template <int NT>
__device__ __forceinline__ uint32_t a_unit(int k, int c) {
  if constexpr (NT >= 8) {
    return (uint32_t)(k * NT + (c ^ (k & 7)));
  } else {
    const uint32_t u = (uint32_t)(k * NT + c);
    return u ^ ((u >> 3) & 7u);
  }
}

// XA[m][j] = sum_k X[m][k] A[k][j] (m < M <= 16, j < r = 8 NT), fp32.  CTA c
// of the cluster takes K rows [k0, k1) (64-aligned) in chunks of at most kcc
// rows.  Per chunk the CTA copies A[chunk][:] (swizzled) and X[m][chunk]
// (rows padded by 16 bytes; rows M..15 stay zero) into shared memory, and
// warp w takes the chunk's 16-wide k steps w, w + 8, ...: X supplies the A
// fragments (16 tokens), A the B fragments (n = j) through transposing loads.
// Warp partials are added in warp order, CTA partials in CTA order.
template <int NT>
__global__ void __launch_bounds__(XA_THREADS)
k_decode_xa(const uint16_t *__restrict__ X, int M, int64_t K, const uint16_t *__restrict__ A, int kcc,
            float *__restrict__ XA, uint16_t *__restrict__ XA_out, int *__restrict__ counters, int n_counters) {
  griddep_launch();
  constexpr int R = NT * 8;
  extern __shared__ __align__(128) uint8_t xa_smem[];
  float *part = reinterpret_cast<float *>(xa_smem);  // [16][128] this CTA's partial
  uint8_t *stage = xa_smem + 16 * 128 * 4;
  const int XS = kcc + 8;                            // X row stride (elements)
  uint16_t *as = reinterpret_cast<uint16_t *>(stage);                       // kcc x R, swizzled units
  uint16_t *xs = reinterpret_cast<uint16_t *>(stage + (size_t)kcc * R * 2);  // 16 x XS
  float *wpart = reinterpret_cast<float *>(stage);   // [warps][16][R], after the last chunk
  const uint32_t crank = ptx::cluster_ctarank(), csize = ptx::cluster_nctarank();
  const int64_t nb = K / 64;
  const int64_t k0 = (int64_t)crank * nb / csize * 64, k1 = (int64_t)(crank + 1) * nb / csize * 64;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  // rows M..15 of the X stage are zero for the whole kernel
  for (int i = tid; i < (16 - M) * XS / 8; i += XA_THREADS)
    reinterpret_cast<uint4 *>(xs + (size_t)M * XS)[i] = make_uint4(0, 0, 0, 0);
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
  const uint32_t as_u = ptx::smem_u32(as), xs_u = ptx::smem_u32(xs);
#pragma unroll 1
  for (int64_t c0 = k0; c0 < k1; c0 += kcc) {
    const int n = (int)min((int64_t)kcc, k1 - c0);
    {  // stage: A rows [c0, c0 + n) and X[m][c0 : c0 + n], 16-byte units, 8 loads in flight per thread
      const int ua = n * NT, ux = M * (n / 8);
      const uint4 *ga = reinterpret_cast<const uint4 *>(A + c0 * R);
#pragma unroll 1
      for (int base = 0; base < ua + ux; base += 8 * XA_THREADS) {
        uint4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int u = base + q * XA_THREADS + tid;
          if (u < ua) {
            v[q] = __ldg(ga + u);
          } else if (u < ua + ux) {
            const int w = u - ua, m = w / (n / 8), c = w - m * (n / 8);
            v[q] = __ldg(reinterpret_cast<const uint4 *>(X + m * K + c0) + c);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int u = base + q * XA_THREADS + tid;
          if (u < ua) {
            reinterpret_cast<uint4 *>(as)[a_unit<NT>(u / NT, u % NT)] = v[q];
          } else if (u < ua + ux) {
            const int w = u - ua, m = w / (n / 8), c = w - m * (n / 8);
            reinterpret_cast<uint4 *>(xs + (size_t)m * XS)[c] = v[q];
          }
        }
      }
    }
    __syncthreads();
#pragma unroll 1
    for (int ks = warp; ks < n / 16; ks += XA_WARPS) {
      uint32_t a0, a1, a2, a3;
      {
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8, col = ks * 16 + (lane >> 4) * 8;
        ldsm_x4(xs_u + (uint32_t)(row * XS + col) * 2u, a0, a1, a2, a3);
      }
      const int kr = ks * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
      if constexpr (NT == 1) {
        uint32_t b0, b1;
        ldsm_x2_t(as_u + a_unit<NT>(kr, 0) * 16u, b0, b1);
        mma16816(acc[0], a0, a1, a2, a3, b0, b1);
      } else {
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(as_u + a_unit<NT>(kr, 2 * np + (lane >> 4)) * 16u, b0, b1, b2, b3);
          mma16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
          mma16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();  // the next chunk (or the warp partials) overwrite the stage
  }
  // warp partials: rows = tokens g, g + 8; columns j = 8 nt + 2t, +1
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float *w = wpart + (size_t)warp * 16 * R + nt * 8 + 2 * t;
    *reinterpret_cast<float2 *>(w + g * R) = make_float2(acc[nt][0], acc[nt][1]);
    *reinterpret_cast<float2 *>(w + (g + 8) * R) = make_float2(acc[nt][2], acc[nt][3]);
  }
  __syncthreads();
  for (int i = tid; i < 16 * R; i += XA_THREADS) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < XA_WARPS; ++w) s += wpart[w * 16 * R + i];
    part[(i / R) * 128 + (i % R)] = s;
  }
  ptx::cluster_sync();
  if (crank == 0) {
    const uint32_t local = ptx::smem_u32(part);
    for (int i = tid; i < M * R; i += XA_THREADS) {
      const int m = i / R, jj = i - m * R;
      float s = 0.0f;
      for (uint32_t c = 0; c < csize; ++c) {
        float v;
        asm volatile("ld.shared::cluster.f32 %0, [%1];"
                     : "=f"(v)
                     : "r"(ptx::mapa(local + (uint32_t)(m * 128 + jj) * 4u, c))
                     : "memory");
        s += v;
      }
      XA[i] = s;
      if (XA_out) XA_out[i] = (uint16_t)(pack_bf16x2(s, 0.0f) & 0xFFFFu);
    }
    for (int i = tid; i < n_counters; i += XA_THREADS) counters[i] = 0;
  }
  // keep every CTA's shared memory alive until CTA 0 has read it
  ptx::cluster_sync();
}

// ---------------------------------------------------------------------------- weight stream
struct StreamArgs {
  const uint16_t *X;
  int M;
  int64_t K;
  const int8_t *code;
  const float *step;
  const float *mean;
  const float *absmax;
  int64_t N;
  int64_t tiles;  // ceil(N / 16)
  int P;          // pieces (warps) per row tile
  float *part;    // [tiles][P][16 rows][16 tokens]
  int *counters;  // [tiles]
  const float *XA;
  const uint16_t *B;
  int r;
  float scale;
  uint16_t *Y;
  int *status;
  float q[16];
};

// Block constants of one box (up to 4 blocks) for rows g and g + 8.  Double
// quantization: w[h][0] = the 4 int8 codes, w[h][1], w[h][2] = the fp32 step
// of the first and of the last block (a box spans at most two groups of 256
// blocks).  Otherwise w[h][0..3] = the 4 fp32 absmax values.
struct BoxC {
  uint32_t w[2][4];
};

template <int MT, bool DQ>  // MT token tiles of 8
__global__ void __launch_bounds__(ST_THREADS, 2)
k_decode_stream(const __grid_constant__ CUtensorMap tmP, const StreamArgs a) {
  griddep_launch();
  extern __shared__ uint8_t smem_raw[];
  __shared__ int last_flag[ST_WARPS];
  __shared__ int abort_flag;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *rings = smem;                                             // [warps][RING][16 x 128 B]
  uint32_t *tab = reinterpret_cast<uint32_t *>(rings + ST_WARPS * RING * BOX_BYTES);  // [256][32 lanes]
  uint64_t *bars = reinterpret_cast<uint64_t *>(tab + 256 * 32);    // [warps][RING]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    // element 2j (high nibble) goes to the low half: it is the lower k of the MMA pair
    const uint32_t v = pack_bf16x2(a.q[(tid >> 4) & 15], a.q[tid & 15]);
    uint4 *dst = reinterpret_cast<uint4 *>(&tab[tid * 32]);
#pragma unroll
    for (int c = 0; c < 8; ++c) dst[c] = make_uint4(v, v, v, v);
  }
  if (lane == 0) {
    for (int s = 0; s < RING; ++s) ptx::mbar_init(ptx::smem_u32(&bars[warp * RING + s]), 1);
    ptx::fence_mbar_init();
  }
  if (tid == 0) abort_flag = 0;
  __syncthreads();

  const int64_t item = (int64_t)blockIdx.x * ST_WARPS + warp;
  const bool active = item < a.tiles * a.P;
  const int64_t rt = active ? item / a.P : 0;
  const int piece = active ? (int)(item - rt * a.P) : 0;
  const int64_t nbox = (a.K + BOX_K - 1) / BOX_K, nb_row = a.K >> 6;
  const int64_t bx0 = piece * nbox / a.P, bx1 = active ? (piece + 1) * nbox / a.P : bx0;
  const int nmine = (int)(bx1 - bx0);
  const int64_t kend = min(bx1 * 4, nb_row);  // one past the warp's last 64-block
  const int g = lane >> 2, t = lane & 3;
  const int64_t rowg = rt * 16 + g, rowg8 = rowg + 8;
  const bool vg = rowg < a.N, vg8 = rowg8 < a.N;
  const uint32_t ring = ptx::smem_u32(rings + warp * RING * BOX_BYTES);
  const uint32_t tl = ptx::smem_u32(tab) + (uint32_t)lane * 4u;
  const float mu = DQ ? __ldg(a.mean) : 0.0f;
  auto bar = [&](int s) { return ptx::smem_u32(&bars[warp * RING + s]); };
  auto issue = [&](int i) {  // lane 0: box bx0 + i into slot i % RING
    const int s = i % RING;
    ptx::mbar_arrive_expect_tx(bar(s), BOX_BYTES);
    ptx::tma_load_2d(ring + s * BOX_BYTES, &tmP, bar(s), (int)((bx0 + i) * 128), (int)(rt * 16));
  };
  if (lane == 0)
    for (int i = 0; i < RING && i < nmine; ++i) issue(i);

  auto load_box = [&](int b) {
    BoxC c;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) c.w[h][e] = 0u;
    if (b >= nmine) return c;
    const int64_t kb0 = (bx0 + b) * 4;
    const bool whole = kb0 + 3 < nb_row && (nb_row & 3) == 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (!(h ? vg8 : vg)) continue;
      const int64_t base = (h ? rowg8 : rowg) * nb_row + kb0;
      if constexpr (DQ) {
        if (whole) {
          c.w[h][0] = __ldg(reinterpret_cast<const uint32_t *>(a.code + base));
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (kb0 + e < nb_row) c.w[h][0] |= (uint32_t)(uint8_t)__ldg(a.code + base + e) << (8 * e);
        }
        c.w[h][1] = __float_as_uint(__ldg(a.step + (base >> 8)));
        c.w[h][2] = __float_as_uint(__ldg(a.step + ((base + min((int64_t)3, nb_row - 1 - kb0)) >> 8)));
      } else {
        if (whole) {
          const float4 v = __ldg(reinterpret_cast<const float4 *>(a.absmax + base));
          c.w[h][0] = __float_as_uint(v.x); c.w[h][1] = __float_as_uint(v.y);
          c.w[h][2] = __float_as_uint(v.z); c.w[h][3] = __float_as_uint(v.w);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (kb0 + e < nb_row) c.w[h][e] = __float_as_uint(__ldg(a.absmax + base + e));
        }
      }
    }
    return c;
  };

  const uint16_t *xr[MT];
  bool xv[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int tok = mt * 8 + g;
    xv[mt] = tok < a.M;
    xr[mt] = a.X + (xv[mt] ? tok : 0) * a.K + t * 16;
  }
  auto load_x = [&](int64_t kb, uint4 (&dst)[MT][2]) {  // this lane's 16 X values of block kb, per token tile
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const uint4 *src = reinterpret_cast<const uint4 *>(xr[mt] + kb * 64);
      dst[mt][0] = xv[mt] ? __ldg(src) : make_uint4(0, 0, 0, 0);
      dst[mt][1] = xv[mt] ? __ldg(src + 1) : make_uint4(0, 0, 0, 0);
    }
  };
  float acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[mt][i] = 0.0f;
  uint4 xn[MT][2];
  if (nmine > 0) load_x(bx0 * 4, xn);
  BoxC pre[PD];
#pragma unroll
  for (int d = 0; d < PD; ++d) pre[d] = load_box(d);

#pragma unroll 1
  for (int i = 0; i < nmine; ++i) {
    const int s = i % RING;
    const BoxC cur = pre[0];
#pragma unroll
    for (int d = 0; d < PD - 1; ++d) pre[d] = pre[d + 1];
    pre[PD - 1] = load_box(i + PD);
    const int64_t kb_base = (bx0 + i) * 4;  // first 64-block of the box
    // wait for the box (in bounds or zero-filled, so it always lands; the
    // wait is bounded all the same, and a warp that gives up lets the boxes
    // it has in flight land and stops without touching the output)
    if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar(s), (uint32_t)((i / RING) & 1), &abort_flag, a.status))) {
      if (lane == 0)
        for (int z = i; z < nmine && z < i + RING; ++z) drain_wait(bar(z % RING), (uint32_t)((z / RING) & 1));
      return;
    }
    const uint32_t slot = ring + s * BOX_BYTES;
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      const int64_t kb = kb_base + blk;
      if (kb >= kend) break;
      uint4 xc[MT][2];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        xc[mt][0] = xn[mt][0];
        xc[mt][1] = xn[mt][1];
      }
      if (kb + 1 < kend) load_x(kb + 1, xn);
      // block constants of rows g, g + 8
      float mh[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if constexpr (DQ) {
          const int code = (int)(int8_t)(uint8_t)(cur.w[h][0] >> (8 * blk));
          const int64_t row = h ? rowg8 : rowg;
          const bool first = ((row * nb_row + kb) >> 8) == ((row * nb_row + kb_base) >> 8);
          const float st = __uint_as_float(first ? cur.w[h][1] : cur.w[h][2]);
          mh[h] = __fadd_rn(__fmul_rn((float)code, st), mu);
        } else {
          mh[h] = __uint_as_float(cur.w[h][blk]);
        }
      }
      // 8 packed bytes of row r, block blk, lane t: chunk 2 blk + t/2 of the
      // 128-byte row, at position chunk ^ (r mod 8) (128-byte swizzle)
      const uint32_t cb = (uint32_t)(2 * blk + (t >> 1));
      const uint2 wg = lds64(slot + g * 128 + ((cb ^ (uint32_t)g) << 4) + (t & 1) * 8);
      const uint2 wg8 = lds64(slot + (g + 8) * 128 + ((cb ^ (uint32_t)g) << 4) + (t & 1) * 8);
      float D[MT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) D[mt][e] = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // MMA j takes k = 16 t + 4 j + [0, 4) of this block: bytes 2j and 2j+1
        const uint32_t wa = (j >> 1) ? wg.y : wg.x, wb = (j >> 1) ? wg8.y : wg8.x;
        const uint32_t s0 = 0x4440u | (uint32_t)((j & 1) * 2), s1 = s0 + 1;
        const uint32_t a0 = lds32(tl + byte_of(wa, s0) * 128u);
        const uint32_t a2 = lds32(tl + byte_of(wa, s1) * 128u);
        const uint32_t a1 = lds32(tl + byte_of(wb, s0) * 128u);
        const uint32_t a3 = lds32(tl + byte_of(wb, s1) * 128u);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t *xw = reinterpret_cast<const uint32_t *>(&xc[mt][0]);
          mma16816(D[mt], a0, a1, a2, a3, xw[2 * j], xw[2 * j + 1]);
        }
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        acc[mt][0] = fmaf(D[mt][0], mh[0], acc[mt][0]);
        acc[mt][1] = fmaf(D[mt][1], mh[0], acc[mt][1]);
        acc[mt][2] = fmaf(D[mt][2], mh[1], acc[mt][2]);
        acc[mt][3] = fmaf(D[mt][3], mh[1], acc[mt][3]);
      }
    }
    // slot s has been read; refill it with box i + RING
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && i + RING < nmine) issue(i + RING);
  }

  // ---- this warp's 16 x 16 partial -> its slot; the last warp of the tile finishes it
  if (active) {
    float *dst = a.part + item * 256;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      *reinterpret_cast<float2 *>(dst + g * 16 + mt * 8 + 2 * t) = make_float2(acc[mt][0], acc[mt][1]);
      *reinterpret_cast<float2 *>(dst + (g + 8) * 16 + mt * 8 + 2 * t) = make_float2(acc[mt][2], acc[mt][3]);
    }
  }
  // XA and the cleared counters come from k_decode_xa
  griddep_wait();
  if (!active) return;
  __threadfence();
  __syncwarp();
  if (lane == 0) last_flag[warp] = atomicAdd(&a.counters[rt], 1) == a.P - 1;
  __syncwarp();
  if (!last_flag[warp]) return;
  __threadfence();
  // The tile's result, in this lane's MMA accumulator positions (rows g, g+8;
  // tokens 8 mt + 2t, +1): the P partials added in piece order ...
  const float *base = a.part + rt * a.P * 256;
  float sum[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) sum[mt][e] = 0.0f;
#pragma unroll 1
  for (int z0 = 0; z0 < a.P; z0 += 4) {
    float2 u[4][MT][2];
#pragma unroll
    for (int dz = 0; dz < 4; ++dz)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const float *pz = base + (z0 + dz) * 256 + mt * 8 + 2 * t;
        const bool in = z0 + dz < a.P;
        u[dz][mt][0] = in ? __ldcg(reinterpret_cast<const float2 *>(pz + g * 16)) : make_float2(0.0f, 0.0f);
        u[dz][mt][1] = in ? __ldcg(reinterpret_cast<const float2 *>(pz + (g + 8) * 16)) : make_float2(0.0f, 0.0f);
      }
#pragma unroll
    for (int dz = 0; dz < 4; ++dz)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        sum[mt][0] += u[dz][mt][0].x;
        sum[mt][1] += u[dz][mt][0].y;
        sum[mt][2] += u[dz][mt][1].x;
        sum[mt][3] += u[dz][mt][1].y;
      }
  }
  // ... and the LoRA term (XA B)^T for the tile by MMA: weight rows are M,
  // tokens N and the rank k.  B supplies the bf16 A fragments; XA (fp32) is
  // split into bf16 high and low parts, two MMAs, so XA keeps about 16 bits.
  float L[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) L[mt][e] = 0.0f;
  auto bpair = [&](int kr, int64_t row, bool v) -> uint32_t {  // B[kr][row], B[kr + 1][row]
    if (!v || kr >= a.r) return 0u;
    return (uint32_t)__ldg(a.B + (int64_t)kr * a.N + row) | ((uint32_t)__ldg(a.B + (int64_t)(kr + 1) * a.N + row) << 16);
  };
#pragma unroll 1
  for (int kk = 0; kk < a.r; kk += 16) {
    const int k = kk + 2 * t;
    const uint32_t a0 = bpair(k, rowg, vg), a1 = bpair(k, rowg8, vg8);
    const uint32_t a2 = bpair(k + 8, rowg, vg), a3 = bpair(k + 8, rowg8, vg8);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const float *xa = a.XA + (int64_t)(mt * 8 + g) * a.r;
      const float2 x0 = xv[mt] && k < a.r ? __ldcg(reinterpret_cast<const float2 *>(xa + k)) : make_float2(0.0f, 0.0f);
      const float2 x1 =
          xv[mt] && k + 8 < a.r ? __ldcg(reinterpret_cast<const float2 *>(xa + k + 8)) : make_float2(0.0f, 0.0f);
      const uint32_t h0 = pack_bf16x2(x0.x, x0.y), h1 = pack_bf16x2(x1.x, x1.y);
      const uint32_t l0 = pack_bf16x2(x0.x - bf16lo_to_f32(h0), x0.y - bf16hi_to_f32(h0));
      const uint32_t l1 = pack_bf16x2(x1.x - bf16lo_to_f32(h1), x1.y - bf16hi_to_f32(h1));
      mma16816(L[mt], a0, a1, a2, a3, h0, h1);
      mma16816(L[mt], a0, a1, a2, a3, l0, l1);
    }
  }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int tok = mt * 8 + 2 * t + (e & 1);
      const bool v = e & 2 ? vg8 : vg;
      if (tok < a.M && v)
        a.Y[(int64_t)tok * a.N + (e & 2 ? rowg8 : rowg)] =
            (uint16_t)(pack_bf16x2(fmaf(a.scale, L[mt][e], sum[mt][e]), 0.0f) & 0xFFFFu);
    }
  if (lane == 0) a.counters[rt] = 0;
}

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Packed nibbles as a 2-D uint8 tensor [N][K/2], boxes of 16 rows x 128 bytes,
// 128-byte swizzle, zero fill past the end of a row.
int tmap_packed(CUtensorMap *tm, const uint8_t *packed, int64_t N, int64_t K) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return set_error(QL_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
  cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  cuuint32_t box[2] = {128, 16};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(packed), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(QL_ERR_CUDA, "cuTensorMapEncodeTiled (packed) failed (%d)", (int)r);
  return QL_OK;
}

template <int NT>
int launch_xa(const DecodeProblem &p, float *xa, int *counters, int n_counters, cudaStream_t st) {
  // chunk rows: A chunk (kcc x r) + X chunk (16 x (kcc + 8)) within the stage,
  // which also holds the warp partials (8 x 16 x r fp32)
  constexpr int R = NT * 8;
  const int64_t kc_max = ((p.K / 64 + XA_CLUSTER - 1) / XA_CLUSTER) * 64;
  const int64_t stage_max = XA_SMEM_MAX - 16 * 128 * 4;
  const int64_t kcc = std::max<int64_t>(64, std::min<int64_t>(kc_max, (stage_max - 256) / (2 * R + 32) / 64 * 64));
  const size_t stage = std::max<size_t>((size_t)kcc * R * 2 + (size_t)16 * (kcc + 8) * 2, (size_t)XA_WARPS * 16 * R * 4);
  const size_t smem = 16 * 128 * 4 + stage;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    int rc = check_cuda(cudaFuncSetAttribute(k_decode_xa<NT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
                        "decode XA: cluster attribute");
    if (!rc)
      rc = check_cuda(cudaFuncSetAttribute(k_decode_xa<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, XA_SMEM_MAX),
                      "decode XA: shared-memory attribute");
    if (rc) return rc;
    attr_done[dev] = true;
  }
  cudaLaunchConfig_t cx{};
  cx.gridDim = dim3(XA_CLUSTER);
  cx.blockDim = dim3(XA_THREADS);
  cx.dynamicSmemBytes = smem;
  cx.stream = st;
  cudaLaunchAttribute ax[1];
  ax[0].id = cudaLaunchAttributeClusterDimension;
  ax[0].val.clusterDim.x = XA_CLUSTER;
  ax[0].val.clusterDim.y = 1;
  ax[0].val.clusterDim.z = 1;
  cx.attrs = ax;
  cx.numAttrs = 1;
  cudaError_t ex = cudaLaunchKernelEx(&cx, k_decode_xa<NT>, p.X, (int)p.M, p.K, p.A, (int)kcc, xa, p.XA_out,
                                      counters, n_counters);
  count_launch();
  return check_cuda(ex, "decode XA launch");
}

}  // namespace

int decode_splits(int64_t N, int64_t K) {
  // Pieces per 16-row tile: as many as fit one warp each on the GPU (148 SMs x
  // 16 resident warps), at most 16, each with at least 2 boxes of 256 K.
  const int64_t tiles = (N + 15) / 16, nbox = (K + BOX_K - 1) / BOX_K;
  int64_t P = (148 * 16) / tiles;
  P = std::min<int64_t>(P, std::max<int64_t>(1, nbox / 2));
  P = std::min<int64_t>(P, 16);
  return (int)std::max<int64_t>(P, 1);
}

size_t decode_ws(int64_t N, int64_t K, int r) {
  (void)r;
  const size_t tiles = (size_t)((N + 15) / 16);
  return up256(16 * 128 * 4) + up256(tiles * 4) + up256(tiles * (size_t)decode_splits(N, K) * 256 * 4);
}

int launch_decode(const DecodeProblem &p, cudaStream_t st) {
  char *ws = static_cast<char *>(p.ws);
  float *xa = reinterpret_cast<float *>(ws);
  const int64_t tiles = (p.N + 15) / 16;
  int *counters = reinterpret_cast<int *>(ws + up256(16 * 128 * 4));
  float *part = reinterpret_cast<float *>(ws + up256(16 * 128 * 4) + up256((size_t)tiles * 4));
  const int P = decode_splits(p.N, p.K);

  int rc = QL_OK;
  switch (p.r) {
    case 8: rc = launch_xa<1>(p, xa, counters, (int)tiles, st); break;
    case 16: rc = launch_xa<2>(p, xa, counters, (int)tiles, st); break;
    case 32: rc = launch_xa<4>(p, xa, counters, (int)tiles, st); break;
    case 64: rc = launch_xa<8>(p, xa, counters, (int)tiles, st); break;
    case 128: rc = launch_xa<16>(p, xa, counters, (int)tiles, st); break;
    default: return set_error(QL_ERR_UNSUPPORTED, "decode: rank %d", p.r);
  }
  if (rc) return rc;

  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    for (auto fn : {k_decode_stream<1, true>, k_decode_stream<2, true>, k_decode_stream<1, false>,
                    k_decode_stream<2, false>})
      if (!rc)
        rc = check_cuda(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ST_SMEM),
                        "decode stream: shared-memory attribute");
    if (rc) return rc;
    attr_done[dev] = true;
  }
  CUtensorMap tmP;
  rc = tmap_packed(&tmP, p.w.packed, p.N, p.K);
  if (rc) return rc;
  StreamArgs a{};
  a.X = p.X; a.M = (int)p.M; a.K = p.K;
  a.code = p.w.code; a.step = p.w.step; a.mean = p.w.mean; a.absmax = p.w.absmax;
  a.N = p.N; a.tiles = tiles; a.P = P; a.part = part; a.counters = counters;
  a.XA = xa; a.B = p.B; a.r = p.r; a.scale = p.scale; a.Y = p.Y; a.status = device_status_ptr();
  const Codebook &cb = codebook();
  for (int i = 0; i < 16; ++i) a.q[i] = cb.q[i];

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)((tiles * P + ST_WARPS - 1) / ST_WARPS));
  cfg.blockDim = dim3(ST_THREADS);
  cfg.dynamicSmemBytes = ST_SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (p.w.dq)
    e = p.M <= 8 ? cudaLaunchKernelEx(&cfg, k_decode_stream<1, true>, tmP, a)
                 : cudaLaunchKernelEx(&cfg, k_decode_stream<2, true>, tmP, a);
  else
    e = p.M <= 8 ? cudaLaunchKernelEx(&cfg, k_decode_stream<1, false>, tmP, a)
                 : cudaLaunchKernelEx(&cfg, k_decode_stream<2, false>, tmP, a);
  count_launch();
  return check_cuda(e, "decode stream launch");
}

}  // namespace ql
