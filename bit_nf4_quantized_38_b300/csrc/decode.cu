// Decode-sized forward (M <= 16 tokens) of the frozen-NF4 linear with LoRA:
//   Y = X W_hat^T + s (X A) B
// At decode batch sizes the layer is bound by HBM traffic on the packed 4-bit
// weights (0.5 B/param + 1/64 B/param of block codes), so this is a streaming
// GEMV / skinny GEMM, not a tile GEMM.  Four kernels, each launched as a
// programmatic dependent of the one before; the weight stream fits beside
// the XA kernel on every SM, so they run concurrently:
//
//   k_decode_xa      XA = X A by warp MMAs on 8 clusters of 16 small CTAs.  Each
//                    CTA stages its 16-row K steps of A (swizzled so that the
//                    transposing fragment loads never conflict) and of X in
//                    shared memory; the cluster adds its CTAs' tiles in rank
//                    order through distributed shared memory.
//   k_decode_xa_final  one CTA adds the clusters' tiles in cluster order.
//   k_decode_stream  The weight stream, one persistent CTA per SM.  The work
//                    is the list of units (256-row group, 256-wide K box) in
//                    row-group-major order, split evenly over the CTAs (at
//                    most one per SM, at least one unit each).  A
//                    producer warp fills a 3-stage shared-memory ring by TMA:
//                    per unit a 256 x 128 B box of packed nibbles (128-byte
//                    swizzle) and four 64-wide boxes of X (rows past M zero
//                    filled).  Eight consumer warps each own 32 weight rows:
//                    every packed byte (two codes) is looked up in a 256-entry
//                    table of bf16 level pairs kept once per lane in shared
//                    memory (one byte permute forms the lookup address, and
//                    lookups never conflict on a bank); warp MMAs m16n8k16
//                    with weight rows as M and tokens as N accumulate each
//                    64-block in a fresh fp32 tile that is then scaled by the
//                    block constant.  A lane computes the constants of block t
//                    for its 4 rows (codes loaded two units ahead) and the
//                    others get them by shuffle.  When a CTA leaves a row
//                    group it stores its partial tile to the group's slot for
//                    that CTA.
//   k_decode_finish  one warp per 16 rows: adds the row group's slots in CTA
//                    order and s (XA B)^T (warp MMAs, B loaded before the
//                    weight stream ends), and writes Y.
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

// ---- XA kernel
constexpr int XA_CLUSTER = 16;       // non-portable cluster size (B300 allows 16)
constexpr int XA_THREADS = 256;
constexpr int XA_WARPS = XA_THREADS / 32;
constexpr int XA_MAX_CLUSTERS = 8;   // one 16-SM cluster per GPC
constexpr int XA_STAGE_MAX = 24 * 1024;  // A and X chunk; + 8 KB partial tile
// ---- weight stream
constexpr int ST_CONS = 8;                     // consumer warps, 32 rows each
constexpr int ST_THREADS = (ST_CONS + 1) * 32;  // + one producer warp
constexpr int ST_STAGES = 3;
constexpr int UNIT_ROWS = 256;                 // rows per unit
constexpr int UNIT_K = 256;                    // K values per unit (128 packed bytes per row)
constexpr int W_BYTES = UNIT_ROWS * 128;       // packed box of a unit
constexpr int TAB_BYTES = 256 * 256;           // 256 entries x 256 B stride (32 lanes x 4 B used)
constexpr int PD = 2;                          // units of block constants loaded ahead
constexpr int G_MAX = 160;                     // persistent CTAs at most (one per SM)
constexpr int SLOT_FLOATS = UNIT_ROWS * 16;    // partial tile of a row group: 256 rows x 16 tokens

template <int MT>
constexpr int stage_bytes() { return W_BYTES + 4 * (MT * 8) * 128; }
template <int MT>
constexpr size_t stream_smem() { return (size_t)TAB_BYTES + 1024 + (size_t)ST_STAGES * stage_bytes<MT>(); }

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
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Wait for phase `parity` of a barrier for at most `limit_ns`, ignoring any
// abort flag: lets copies already in flight land before a CTA that gave up
// exits.
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

struct XaArgs {
  const uint16_t *X;
  int M;
  int64_t K;
  const uint16_t *A;
  int kcc;          // rows per staged chunk (multiple of 16)
  float *xap;       // [clusters][16][R] cluster partials
  float *XA;        // [M][R] fp32 result
  uint16_t *XA_out; // [M][R] bf16 copy or null
};

// XA[m][j] = sum_k X[m][k] A[k][j] (m < M <= 16, j < R = 8 NT), fp32.  CTA c
// of G takes the 16-row K steps [c KS / G, (c+1) KS / G), KS = K / 16, in
// chunks of kcc rows: it copies A[chunk][:] (swizzled) and X[m][chunk] (rows
// padded by 16 bytes; rows M..15 stay zero) into shared memory.  Warp w owns
// the 8-column tiles w, w + 8 of XA: X supplies the A fragments (16 tokens)
// and A the B fragments (n = j) through transposing loads.
template <int NT>
__global__ void __launch_bounds__(XA_THREADS)
k_decode_xa(const XaArgs a) {
  griddep_launch();
  constexpr int R = NT * 8;
  extern __shared__ __align__(128) uint8_t xa_smem[];
  float *part = reinterpret_cast<float *>(xa_smem);  // [16][128] this CTA's tile
  uint8_t *stage = xa_smem + 16 * 128 * 4;
  const int XS = a.kcc + 8;                          // X row stride (elements)
  uint16_t *as = reinterpret_cast<uint16_t *>(stage);                          // kcc x R, swizzled units
  uint16_t *xs = reinterpret_cast<uint16_t *>(stage + (size_t)a.kcc * R * 2);  // 16 x XS
  const int64_t KS = a.K / 16, G = gridDim.x, c = blockIdx.x;
  const int64_t k0 = c * KS / G * 16, k1 = (c + 1) * KS / G * 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int M = a.M;
  for (int i = tid; i < (16 - M) * XS / 8; i += XA_THREADS)
    reinterpret_cast<uint4 *>(xs + (size_t)M * XS)[i] = make_uint4(0, 0, 0, 0);
  constexpr int NTW = (NT + XA_WARPS - 1) / XA_WARPS;  // column tiles per warp
  float acc[NTW][4];
#pragma unroll
  for (int q = 0; q < NTW; ++q)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[q][e] = 0.0f;
  const uint32_t as_u = ptx::smem_u32(as), xs_u = ptx::smem_u32(xs);
#pragma unroll 1
  for (int64_t c0 = k0; c0 < k1; c0 += a.kcc) {
    const int n = (int)min((int64_t)a.kcc, k1 - c0);
    {  // stage A rows [c0, c0 + n) and X[m][c0 : c0 + n] in 16-byte units, 8 loads in flight per thread
      const int ua = n * NT, ux = M * (n / 8);
      const uint4 *ga = reinterpret_cast<const uint4 *>(a.A + c0 * R);
#pragma unroll 1
      for (int base = 0; base < ua + ux; base += 8 * XA_THREADS) {
        uint4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int u = base + q * XA_THREADS + tid;
          if (u < ua) {
            v[q] = __ldg(ga + u);
          } else if (u < ua + ux) {
            const int w = u - ua, m = w / (n / 8), cc = w - m * (n / 8);
            v[q] = __ldg(reinterpret_cast<const uint4 *>(a.X + m * a.K + c0) + cc);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int u = base + q * XA_THREADS + tid;
          if (u < ua) {
            reinterpret_cast<uint4 *>(as)[a_unit<NT>(u / NT, u % NT)] = v[q];
          } else if (u < ua + ux) {
            const int w = u - ua, m = w / (n / 8), cc = w - m * (n / 8);
            reinterpret_cast<uint4 *>(xs + (size_t)m * XS)[cc] = v[q];
          }
        }
      }
    }
    __syncthreads();
    if (warp < NT) {
#pragma unroll 1
      for (int ks = 0; ks < n / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        {
          const int row = (lane & 7) + ((lane >> 3) & 1) * 8, col = ks * 16 + (lane >> 4) * 8;
          ldsm_x4(xs_u + (uint32_t)(row * XS + col) * 2u, a0, a1, a2, a3);
        }
        const int kr = ks * 16 + (lane & 15);
#pragma unroll
        for (int q = 0; q < NTW; ++q) {
          const int nt = warp + q * XA_WARPS;
          if (nt < NT) {
            uint32_t b0, b1;
            ldsm_x2_t(as_u + a_unit<NT>(kr, nt) * 16u, b0, b1);
            mma16816(acc[q], a0, a1, a2, a3, b0, b1);
          }
        }
      }
    }
    __syncthreads();  // the next chunk overwrites the stage
  }
  // this CTA's tile: rows = tokens g, g + 8; columns j = 8 nt + 2t, +1
#pragma unroll
  for (int q = 0; q < NTW; ++q) {
    const int nt = warp + q * XA_WARPS;
    if (nt < NT) {
      *reinterpret_cast<float2 *>(part + g * 128 + nt * 8 + 2 * t) = make_float2(acc[q][0], acc[q][1]);
      *reinterpret_cast<float2 *>(part + (g + 8) * 128 + nt * 8 + 2 * t) = make_float2(acc[q][2], acc[q][3]);
    }
  }
  ptx::cluster_sync();
  const uint32_t crank = ptx::cluster_ctarank(), csize = ptx::cluster_nctarank();
  const int64_t cl = c / csize, ncl = G / csize;
  if (crank == 0) {
    const uint32_t local = ptx::smem_u32(part);
    for (int i = tid; i < M * R; i += XA_THREADS) {
      const int m = i / R, jj = i - m * R;
      float v[XA_CLUSTER];  // every CTA's value loaded before adding, in rank order
#pragma unroll
      for (uint32_t cc = 0; cc < XA_CLUSTER; ++cc) {
        v[cc] = 0.0f;
        if (cc < csize)
          asm volatile("ld.shared::cluster.f32 %0, [%1];"
                       : "=f"(v[cc])
                       : "r"(ptx::mapa(local + (uint32_t)(m * 128 + jj) * 4u, cc))
                       : "memory");
      }
      float s = 0.0f;
#pragma unroll
      for (uint32_t cc = 0; cc < XA_CLUSTER; ++cc)
        if (cc < csize) s += v[cc];
      a.xap[cl * 16 * R + i] = s;
    }
  }
  (void)ncl;
  // keep every CTA's shared memory alive until rank 0 has read it
  ptx::cluster_sync();
}

// XA = the clusters' tiles added in cluster order (one CTA, a programmatic
// dependent of k_decode_xa), fp32 and, if asked for, bf16.
constexpr int XF_THREADS = 256;
__global__ void __launch_bounds__(XF_THREADS)
k_decode_xa_final(const XaArgs a, int R, int ncl) {
  griddep_launch();
  griddep_wait();
  const int tid = threadIdx.x, n = a.M * R;
#pragma unroll 1
  for (int i0 = 0; i0 < n; i0 += 4 * XF_THREADS) {
    float v[4][XA_MAX_CLUSTERS];  // 4 outputs per thread, every cluster's tile loaded before adding
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int z = 0; z < XA_MAX_CLUSTERS; ++z) {
        const int i = i0 + q * XF_THREADS + tid;
        v[q][z] = z < ncl && i < n ? __ldcg(a.xap + (int64_t)z * 16 * R + i) : 0.0f;
      }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = i0 + q * XF_THREADS + tid;
      float s = 0.0f;
#pragma unroll
      for (int z = 0; z < XA_MAX_CLUSTERS; ++z)
        if (z < ncl) s += v[q][z];
      if (i < n) {
        a.XA[i] = s;
        if (a.XA_out) a.XA_out[i] = (uint16_t)(pack_bf16x2(s, 0.0f) & 0xFFFFu);
      }
    }
  }
}

// ---------------------------------------------------------------------------- weight stream
struct StreamArgs {  // N K / 64 < 2^31 and units < 2^31 (checked on the host)
  int M;
  int K, N;
  const int8_t *code;
  const float *step;
  const float *mean;
  const float *absmax;
  int nbox;       // ceil(K / 256)
  int W;          // units = row groups x nbox
  float *slots;   // [row groups + G][256 rows][16 tokens]
  int *status;
  float q[16];
};

template <int MT, bool DQ>  // MT token tiles of 8
__global__ void __launch_bounds__(ST_THREADS, 1)
k_decode_stream(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const StreamArgs a) {
  constexpr int XR = MT * 8, SB = stage_bytes<MT>();
  griddep_launch();
  extern __shared__ __align__(16) uint8_t st_smem[];
  __shared__ uint64_t full_bar[ST_STAGES], empty_bar[ST_STAGES];
  __shared__ int abort_flag;
  volatile int *abort_v = &abort_flag;
  const uint32_t tab = ptx::smem_u32(st_smem);  // the lookup table sits at the start
  const uint32_t stages = (tab + TAB_BYTES + 1023u) & ~1023u;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    // entry e (a packed byte), lane l: bf16 pair (q[e >> 4], q[e & 15]); the
    // high nibble is element 2j, the lower k of the MMA pair, in the low half
    uint4 *tp = reinterpret_cast<uint4 *>(st_smem);
    for (int i = tid; i < 256 * 8; i += ST_THREADS) {
      const uint32_t v = pack_bf16x2(a.q[(i >> 7) & 15], a.q[(i >> 3) & 15]);
      tp[(i >> 3) * 16 + (i & 7)] = make_uint4(v, v, v, v);
    }
  }
  if (tid == 0) {
    for (int s = 0; s < ST_STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), ST_CONS);
    }
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();

  const int G = gridDim.x, c = blockIdx.x;
  const int u0 = (int)((int64_t)c * a.W / G), u1 = (int)((int64_t)(c + 1) * a.W / G);
  const int nu = u1 - u0;
  const int nb_row = a.K >> 6;
  const int rg0 = u0 / a.nbox, b0 = u0 - rg0 * a.nbox;  // first unit's row group and K box

  if (warp == ST_CONS) {
    // ---- producer: one lane issues the TMA loads of the ring
    if (lane == 0) {
      ptx::prefetch_tmap(&tmW);
      ptx::prefetch_tmap(&tmX);
      int rg = rg0, b = b0;
      for (int i = 0; i < nu; ++i, b = b + 1 == a.nbox ? 0 : b + 1, rg += b == 0) {
        const int s = i % ST_STAGES;
        if (i >= ST_STAGES &&
            !ptx::mbar_wait(ptx::smem_u32(&empty_bar[s]), (uint32_t)((i / ST_STAGES - 1) & 1), abort_v,
                            a.status))
          break;
        const uint32_t fb = ptx::smem_u32(&full_bar[s]), dst = stages + (uint32_t)(s * SB);
        ptx::mbar_arrive_expect_tx(fb, (uint32_t)SB);
        ptx::tma_load_2d(dst, &tmW, fb, b * 128, rg * UNIT_ROWS);
#pragma unroll
        for (int j = 0; j < 4; ++j) ptx::tma_load_2d(dst + W_BYTES + j * XR * 128, &tmX, fb, b * UNIT_K + 64 * j, 0);
      }
    }
    return;
  }

  // ---- consumers: warp w owns rows 32 w .. 32 w + 31 of the unit's row group
  const int g = lane >> 2, t = lane & 3;
  const uint32_t lanebase = (uint32_t)lane * 4u;
  const float mu = DQ ? __ldg(a.mean) : 0.0f;
  // rows of this lane: k = 0..3 -> 32 w + 16 (k >> 1) + 8 (k & 1) + g
  auto row_of = [&](int k) { return warp * 32 + 16 * (k >> 1) + 8 * (k & 1) + g; };

  // block constants of block t of a unit for the lane's 4 rows, loaded PD units ahead
  struct Pre {
    float a[4], b[4];
  };
  int prg = rg0, pb = b0;  // unit of the next load_pre call
  auto load_pre = [&](int i) {
    Pre p;
#pragma unroll
    for (int k = 0; k < 4; ++k) p.a[k] = p.b[k] = 0.0f;
    const int rg = prg, kb = pb * 4 + t;
    pb = pb + 1 == a.nbox ? 0 : pb + 1;
    prg += pb == 0;
    if (i >= nu || kb >= nb_row) return p;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int row = rg * UNIT_ROWS + row_of(k);
      if (row < a.N) {
        const int bi = row * nb_row + kb;
        if constexpr (DQ) {
          p.a[k] = (float)__ldg(a.code + bi);
          p.b[k] = __ldg(a.step + (bi >> 8));
        } else {
          p.a[k] = __ldg(a.absmax + bi);
        }
      }
    }
    return p;
  };
  Pre pre[PD];
#pragma unroll
  for (int d = 0; d < PD; ++d) pre[d] = load_pre(d);

  float acc[2][MT][4];
  auto zero_acc = [&]() {
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[tt][mt][e] = 0.0f;
  };
  zero_acc();

  // Leave row group rg: store this CTA's partial tile to slot rg + c
  // (k_decode_finish adds the group's slots).
  auto flush = [&](int rg) {
    float *slot = a.slots + (int64_t)(rg + c) * SLOT_FLOATS;
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int rl = warp * 32 + tt * 16 + g;
        *reinterpret_cast<float2 *>(slot + rl * 16 + mt * 8 + 2 * t) = make_float2(acc[tt][mt][0], acc[tt][mt][1]);
        *reinterpret_cast<float2 *>(slot + (rl + 8) * 16 + mt * 8 + 2 * t) =
            make_float2(acc[tt][mt][2], acc[tt][mt][3]);
      }
    zero_acc();
  };

  int cur_rg = -1, rg = rg0, b = b0;
#pragma unroll 1
  for (int i = 0; i < nu; ++i, b = b + 1 == a.nbox ? 0 : b + 1, rg += b == 0) {
    const int s = i % ST_STAGES;
    if (rg != cur_rg) {
      if (cur_rg >= 0) flush(cur_rg);
      cur_rg = rg;
    }
    // block constants of block t of this unit, rows k = 0..3
    float mh[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      mh[k] = DQ ? __fadd_rn(__fmul_rn(pre[0].a[k], pre[0].b[k]), mu) : pre[0].a[k];
#pragma unroll
    for (int d = 0; d < PD - 1; ++d) pre[d] = pre[d + 1];
    pre[PD - 1] = load_pre(i + PD);

    bool landed = false;
    if (!*abort_v)
      landed = ptx::mbar_wait(ptx::smem_u32(&full_bar[s]), (uint32_t)((i / ST_STAGES) & 1), abort_v, a.status);
    const bool ok = __all_sync(0xffffffffu, landed);
    if (ok) {
      const uint32_t wsb = stages + (uint32_t)(s * SB), xsb = wsb + W_BYTES;
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        if (b * 4 + blk >= nb_row) break;
        // X fragments of block blk: token rows 8 mt + g, K values 16 t .. 16 t + 15
        // (16-byte chunks 2t, 2t+1 of the 128-byte row, swizzled by row mod 8)
        uint32_t xw[MT][8];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t rowa = xsb + (uint32_t)(blk * XR * 128 + (mt * 8 + g) * 128);
          const uint4 x0 = lds128(rowa + ((uint32_t)((2 * t) ^ g) << 4));
          const uint4 x1 = lds128(rowa + ((uint32_t)((2 * t + 1) ^ g) << 4));
          xw[mt][0] = x0.x; xw[mt][1] = x0.y; xw[mt][2] = x0.z; xw[mt][3] = x0.w;
          xw[mt][4] = x1.x; xw[mt][5] = x1.y; xw[mt][6] = x1.z; xw[mt][7] = x1.w;
        }
        float m4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) m4[k] = __shfl_sync(0xffffffffu, mh[k], (g << 2) | blk);
        // packed bytes of block blk, lane t: chunk 2 blk + t/2 of the row, at
        // position chunk ^ (row mod 8) (128-byte swizzle), 8 bytes
        const uint32_t coff = ((uint32_t)((2 * blk + (t >> 1)) ^ g) << 4) + (uint32_t)(t & 1) * 8u;
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
          const uint32_t r0 = wsb + (uint32_t)(warp * 32 + tt * 16 + g) * 128u + coff;
          const uint2 wg = lds64(r0), wg8 = lds64(r0 + 8 * 128);
          float D[MT][4];
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) D[mt][e] = 0.0f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // MMA j takes k = 16 t + 4 j + [0, 4) of this block: bytes 2j and 2j+1
            const uint32_t wa = (j >> 1) ? wg.y : wg.x, wb = (j >> 1) ? wg8.y : wg8.x;
            const uint32_t s0 = 0x5504u | ((uint32_t)((j & 1) * 2) << 4), s1 = s0 + 0x10u;
            const uint32_t a0 = lds32(tab + prmt(wa, lanebase, s0));
            const uint32_t a2 = lds32(tab + prmt(wa, lanebase, s1));
            const uint32_t a1 = lds32(tab + prmt(wb, lanebase, s0));
            const uint32_t a3 = lds32(tab + prmt(wb, lanebase, s1));
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) mma16816(D[mt], a0, a1, a2, a3, xw[mt][2 * j], xw[mt][2 * j + 1]);
          }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            acc[tt][mt][0] = fmaf(D[mt][0], m4[2 * tt], acc[tt][mt][0]);
            acc[tt][mt][1] = fmaf(D[mt][1], m4[2 * tt], acc[tt][mt][1]);
            acc[tt][mt][2] = fmaf(D[mt][2], m4[2 * tt + 1], acc[tt][mt][2]);
            acc[tt][mt][3] = fmaf(D[mt][3], m4[2 * tt + 1], acc[tt][mt][3]);
          }
        }
      }
    }
    // stage s has been read
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&empty_bar[s]));
  }
  if (cur_rg >= 0) flush(cur_rg);
  // this grid completes only after the XA kernels it depends on, so the
  // finishing kernel (a dependent of this one) may read XA
  if (tid == 0) griddep_wait();
  // a CTA that gave up lets the loads it still has in flight land before exiting
  if (*abort_v && tid == 0)
    for (int i = std::max(0, nu - ST_STAGES); i < nu; ++i)
      drain_wait(ptx::smem_u32(&full_bar[i % ST_STAGES]), (uint32_t)((i / ST_STAGES) & 1));
}

// ---------------------------------------------------------------------------- finish
struct FinArgs {
  int M, N;
  int nbox, W, G;       // the weight stream's unit split
  const float *slots;   // its partial tiles
  const float *XA;      // [M][R] fp32
  const uint16_t *B;    // [R][N]
  float scale;
  uint16_t *Y;
};
constexpr int FIN_WARPS = 4;

__device__ __forceinline__ uint32_t movtrans(uint32_t v) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(v));
  return r;
}

// Y = bf16(main term + s (XA B)^T), one warp per 16-row tile.  Before waiting
// for the weight stream the warp loads its B[:, rows] fragments (B is an
// input): 8 x 8 blocks read row-wise, 4 bytes per lane, and transposed in
// registers, which gives MMA A fragments with weight rows as M and the rank
// as k.  After the wait it adds the row group's partial tiles in CTA order
// and runs the LoRA MMAs with XA (fp32, split into bf16 high and low parts, so
// XA keeps about 16 bits) as the B fragments, tokens as N.
template <int MT, int R>
__global__ void __launch_bounds__(FIN_WARPS * 32)
k_decode_finish(const FinArgs a) {
  constexpr int KS = (R + 15) / 16;
  constexpr int ZB = MT == 1 ? 8 : 4;  // partial tiles loaded per batch
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int tile = blockIdx.x * FIN_WARPS + warp;
  const bool live = tile * 16 < a.N;  // N % 8 == 0: rows g of a live tile are valid
  const int row0 = tile * 16;
  uint32_t af[KS][4];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int f = 0; f < 4; ++f) {  // a0: (rows 0-7, k 0-7), a1: rows 8-15, a2: k 8-15, a3: both
      const int k = ks * 16 + 8 * (f >> 1) + g, n = row0 + 8 * (f & 1) + 2 * t;
      af[ks][f] = (live && k < R && n < a.N) ? __ldg(reinterpret_cast<const uint32_t *>(a.B + (int64_t)k * a.N + n))
                                             : 0u;
    }
  griddep_wait();  // the weight stream, and through it the XA kernels, completed
  if (!live) return;
  const int rg = tile >> 4, rl = (tile & 15) * 16 + g;
  const int rowg = row0 + g, rowg8 = rowg + 8;
  const bool vg8 = rowg8 < a.N;
  // CTAs of the stream that worked on row group rg: cta(u) = floor(((u+1) G - 1) / W)
  const int cf = (int)((((int64_t)rg * a.nbox + 1) * a.G - 1) / a.W);
  const int cl = (int)((((int64_t)(rg + 1) * a.nbox) * a.G - 1) / a.W);
  const float *base = a.slots + (int64_t)(rg + cf) * SLOT_FLOATS;
  // XA fragments: token 8 mt + g, k pairs (16 ks + 2t, +1) and (+8, +9).
  // Every warp reads the same few lines: through L1 (read-only from here on),
  // so that each SM asks L2 for them once instead of every warp.
  float2 xf[KS][MT][2];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int k = ks * 16 + 2 * t;
      const bool tv = mt * 8 + g < a.M;
      const float *xa = a.XA + (mt * 8 + g) * R;
      xf[ks][mt][0] = tv && k < R ? __ldg(reinterpret_cast<const float2 *>(xa + k)) : make_float2(0.0f, 0.0f);
      xf[ks][mt][1] = tv && k + 8 < R ? __ldg(reinterpret_cast<const float2 *>(xa + k + 8)) : make_float2(0.0f, 0.0f);
    }
  float2 sm[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) sm[mt][0] = sm[mt][1] = make_float2(0.0f, 0.0f);
#pragma unroll 1
  for (int z0 = 0; z0 <= cl - cf; z0 += ZB) {
    float2 v[ZB][MT][2];
#pragma unroll
    for (int dz = 0; dz < ZB; ++dz)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const bool in = z0 + dz <= cl - cf;
        const float *pz = base + (int64_t)(z0 + dz) * SLOT_FLOATS + mt * 8 + 2 * t;
        v[dz][mt][0] = in ? __ldcg(reinterpret_cast<const float2 *>(pz + rl * 16)) : make_float2(0.0f, 0.0f);
        v[dz][mt][1] = in ? __ldcg(reinterpret_cast<const float2 *>(pz + (rl + 8) * 16)) : make_float2(0.0f, 0.0f);
      }
#pragma unroll
    for (int dz = 0; dz < ZB; ++dz)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          sm[mt][h].x += v[dz][mt][h].x;
          sm[mt][h].y += v[dz][mt][h].y;
        }
  }
  float L[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) L[mt][e] = 0.0f;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const uint32_t a0 = movtrans(af[ks][0]), a1 = movtrans(af[ks][1]);
    const uint32_t a2 = movtrans(af[ks][2]), a3 = movtrans(af[ks][3]);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const float2 x0 = xf[ks][mt][0], x1 = xf[ks][mt][1];
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
      const float m = (e & 1) ? sm[mt][e >> 1].y : sm[mt][e >> 1].x;
      if (tok < a.M && ((e & 2) ? vg8 : true))
        a.Y[(int64_t)tok * a.N + ((e & 2) ? rowg8 : rowg)] =
            (uint16_t)(pack_bf16x2(fmaf(a.scale, L[mt][e], m), 0.0f) & 0xFFFFu);
    }
}

constexpr size_t up256(size_t x) { return (x + 255) / 256 * 256; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Packed nibbles as a 2-D uint8 tensor [N][K/2], boxes of 256 rows x 128 bytes;
// X as a 2-D bf16 tensor [M][K], boxes of XR rows x 64 values.  Both 128-byte
// swizzled, zero fill outside the tensor.
int make_tmaps(CUtensorMap *tw, CUtensorMap *tx, const uint8_t *packed, int64_t N, int64_t K, const uint16_t *X,
               int64_t M, int XR) {
  auto fn = encode_fn();
  if (!fn) return set_error(QL_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  {
    cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {128, UNIT_ROWS};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(packed), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(QL_ERR_CUDA, "cuTensorMapEncodeTiled (packed) failed (%d)", (int)r);
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)XR};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(X), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(QL_ERR_CUDA, "cuTensorMapEncodeTiled (X) failed (%d)", (int)r);
  }
  return QL_OK;
}

struct DevInfo {
  int sms = 0;
  bool xa_attr[5] = {};
  bool st_attr = false;
};
DevInfo &dev_info(int dev) {
  static DevInfo info[64];
  return info[dev & 63];
}

// workspace layout
constexpr size_t WS_XA = 0;
constexpr size_t WS_XAP = up256(16 * 128 * 4);
constexpr size_t WS_SLOTS = WS_XAP + up256((size_t)XA_MAX_CLUSTERS * 16 * 128 * 4);

template <typename F>
int max_carveout(F *fn) {
  return check_cuda(cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared),
                    "decode: shared-memory carveout");
}

template <int NT>
int launch_xa(const DecodeProblem &p, char *ws, int sms, DevInfo &di, int ti, cudaStream_t st) {
  const int64_t groups = (p.N + UNIT_ROWS - 1) / UNIT_ROWS;
  (void)groups;
  constexpr int R = NT * 8;
  // chunk rows: A chunk (kcc x R) + X chunk (16 x (kcc + 8)) within XA_STAGE_MAX
  const int GX = XA_MAX_CLUSTERS * XA_CLUSTER;  // 128 CTAs: one cluster per GPC

  const int64_t steps_max = (p.K / 16 + GX - 1) / GX;
  const int64_t kcc = std::max<int64_t>(
      16, std::min<int64_t>(steps_max * 16, (XA_STAGE_MAX - 256) / (2 * R + 32) / 16 * 16));
  const size_t smem = 16 * 128 * 4 + (size_t)kcc * R * 2 + (size_t)16 * (kcc + 8) * 2;
  if (!di.xa_attr[ti]) {
    int rc = check_cuda(cudaFuncSetAttribute(k_decode_xa<NT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
                        "decode XA: cluster attribute");
    if (!rc)
      rc = check_cuda(cudaFuncSetAttribute(k_decode_xa<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           16 * 128 * 4 + XA_STAGE_MAX + 1024),
                      "decode XA: shared-memory attribute");
    // Every decode kernel asks for the largest shared-memory carveout: an SM
    // configured for a small one could not take a weight-stream CTA beside it.
    if (!rc) rc = max_carveout(k_decode_xa<NT>);
    if (!rc) rc = max_carveout(k_decode_xa_final);
    if (!rc) rc = max_carveout(k_decode_finish<1, R>);
    if (!rc) rc = max_carveout(k_decode_finish<2, R>);
    if (rc) return rc;
    di.xa_attr[ti] = true;
  }
  XaArgs a{};
  a.X = p.X; a.M = (int)p.M; a.K = p.K; a.A = p.A; a.kcc = (int)kcc;
  a.xap = reinterpret_cast<float *>(ws + WS_XAP);
  a.XA = reinterpret_cast<float *>(ws + WS_XA);
  a.XA_out = p.XA_out;
  cudaLaunchConfig_t cx{};
  cx.gridDim = dim3(GX);
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
  cudaError_t ex = cudaLaunchKernelEx(&cx, k_decode_xa<NT>, a);
  count_launch();
  int rc = check_cuda(ex, "decode XA launch");
  if (rc) return rc;
  cudaLaunchConfig_t cf{};
  cf.gridDim = dim3(1);
  cf.blockDim = dim3(XF_THREADS);
  cf.stream = st;
  cudaLaunchAttribute af[1];
  af[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  af[0].val.programmaticStreamSerializationAllowed = 1;
  cf.attrs = af;
  cf.numAttrs = 1;
  ex = cudaLaunchKernelEx(&cf, k_decode_xa_final, a, R, GX / XA_CLUSTER);
  count_launch();
  return check_cuda(ex, "decode XA final launch");
}

}  // namespace

size_t decode_ws(int64_t N, int64_t K, int r) {
  (void)K;
  (void)r;
  const size_t groups = (size_t)((N + UNIT_ROWS - 1) / UNIT_ROWS);
  return WS_SLOTS + (groups + G_MAX) * SLOT_FLOATS * 4;
}

int launch_decode(const DecodeProblem &p, cudaStream_t st) {
  char *ws = static_cast<char *>(p.ws);
  const int64_t groups = (p.N + UNIT_ROWS - 1) / UNIT_ROWS;
  float *slots = reinterpret_cast<float *>(ws + WS_SLOTS);
  int dev = 0;
  int rc = check_cuda(cudaGetDevice(&dev), "decode: current device");
  if (rc) return rc;
  DevInfo &di = dev_info(dev);
  if (!di.sms) {
    rc = check_cuda(cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev), "decode: SM count");
    if (rc) return rc;
  }

  switch (p.r) {
    case 8: rc = launch_xa<1>(p, ws, di.sms, di, 0, st); break;
    case 16: rc = launch_xa<2>(p, ws, di.sms, di, 1, st); break;
    case 32: rc = launch_xa<4>(p, ws, di.sms, di, 2, st); break;
    case 64: rc = launch_xa<8>(p, ws, di.sms, di, 3, st); break;
    case 128: rc = launch_xa<16>(p, ws, di.sms, di, 4, st); break;
    default: return set_error(QL_ERR_UNSUPPORTED, "decode: rank %d", p.r);
  }
  if (rc) return rc;

  if (!di.st_attr) {
    rc = check_cuda(cudaFuncSetAttribute(k_decode_stream<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)stream_smem<1>()),
                    "decode stream: shared-memory attribute");
    if (!rc)
      rc = check_cuda(cudaFuncSetAttribute(k_decode_stream<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)stream_smem<1>()),
                      "decode stream: shared-memory attribute");
    if (!rc)
      rc = check_cuda(cudaFuncSetAttribute(k_decode_stream<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)stream_smem<2>()),
                      "decode stream: shared-memory attribute");
    if (!rc)
      rc = check_cuda(cudaFuncSetAttribute(k_decode_stream<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)stream_smem<2>()),
                      "decode stream: shared-memory attribute");
    if (!rc) rc = max_carveout(k_decode_stream<1, true>);
    if (!rc) rc = max_carveout(k_decode_stream<1, false>);
    if (!rc) rc = max_carveout(k_decode_stream<2, true>);
    if (!rc) rc = max_carveout(k_decode_stream<2, false>);

    if (rc) return rc;
    di.st_attr = true;
  }
  const bool mt2 = p.M > 8;
  CUtensorMap tmW, tmX;
  rc = make_tmaps(&tmW, &tmX, p.w.packed, p.N, p.K, p.X, p.M, mt2 ? 16 : 8);
  if (rc) return rc;
  if (p.N * (p.K / 64) >= ((int64_t)1 << 31) || groups * ((p.K + UNIT_K - 1) / UNIT_K) >= ((int64_t)1 << 31))
    return set_error(QL_ERR_UNSUPPORTED, "decode: %lld x %lld weight too large", (long long)p.N, (long long)p.K);
  StreamArgs a{};
  a.M = (int)p.M; a.K = (int)p.K; a.N = (int)p.N;
  a.code = p.w.code; a.step = p.w.step; a.mean = p.w.mean; a.absmax = p.w.absmax;
  a.nbox = (int)((p.K + UNIT_K - 1) / UNIT_K);
  a.W = (int)(groups * a.nbox);
  // every CTA gets at least one unit, so the CTAs of a row group are consecutive
  const int G = (int)std::min<int64_t>(std::min(di.sms, G_MAX), a.W);
  a.slots = slots;
  a.status = device_status_ptr();
  const Codebook &cb = codebook();
  for (int i = 0; i < 16; ++i) a.q[i] = cb.q[i];

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(ST_THREADS);
  cfg.dynamicSmemBytes = mt2 ? stream_smem<2>() : stream_smem<1>();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (p.w.dq)
    e = mt2 ? cudaLaunchKernelEx(&cfg, k_decode_stream<2, true>, tmW, tmX, a)
            : cudaLaunchKernelEx(&cfg, k_decode_stream<1, true>, tmW, tmX, a);
  else
    e = mt2 ? cudaLaunchKernelEx(&cfg, k_decode_stream<2, false>, tmW, tmX, a)
            : cudaLaunchKernelEx(&cfg, k_decode_stream<1, false>, tmW, tmX, a);
  count_launch();
  rc = check_cuda(e, "decode stream launch");
  if (rc) return rc;

  FinArgs f{};
  f.M = (int)p.M; f.N = (int)p.N;
  f.nbox = a.nbox; f.W = a.W; f.G = G;
  f.slots = slots;
  f.XA = reinterpret_cast<const float *>(ws + WS_XA);
  f.B = p.B; f.scale = p.scale; f.Y = p.Y;
  cudaLaunchConfig_t ff{};
  ff.gridDim = dim3((unsigned)(((p.N + 15) / 16 + FIN_WARPS - 1) / FIN_WARPS));
  ff.blockDim = dim3(FIN_WARPS * 32);
  ff.stream = st;
  ff.attrs = attr;
  ff.numAttrs = 1;
  switch (p.r * 4 + (mt2 ? 2 : 1)) {
#define QL_FIN(R_)                                                   \
  case R_ * 4 + 1: e = cudaLaunchKernelEx(&ff, k_decode_finish<1, R_>, f); break; \
  case R_ * 4 + 2: e = cudaLaunchKernelEx(&ff, k_decode_finish<2, R_>, f); break;
    QL_FIN(8) QL_FIN(16) QL_FIN(32) QL_FIN(64) QL_FIN(128)
#undef QL_FIN
    default: return set_error(QL_ERR_UNSUPPORTED, "decode: rank %d", p.r);
  }
  count_launch();
  return check_cuda(e, "decode finish launch");
}

}  // namespace ql
