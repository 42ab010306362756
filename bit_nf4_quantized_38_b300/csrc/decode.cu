// Decode-sized forward (M <= 32 tokens) of the frozen-NF4 linear with LoRA:
//   Y = X W_hat^T + s (X A) B
// At decode batch sizes the layer is bound by HBM traffic on the packed 4-bit
// weights (0.5 B/param + 1/64 B/param of block codes), so this is a streaming
// GEMV / skinny GEMM, not a tile GEMM.  Two kernels per call:
//
//   k_decode_stream  one persistent CTA per SM (at most), 16 warps.  The
//                    units (256-row group x 256-wide K box) are taken in
//                    row-group-major order and split evenly over the CTAs.  A
//                    3-stage (2-stage with 32 tokens) shared-memory ring is
//                    filled by TMA: per unit a 256 x 128 B box of packed
//                    nibbles (128-byte swizzle) and four 64-wide boxes of X
//                    (rows past M zero filled).  The first units are loaded
//                    at the start, each later one by the last warp to finish
//                    with a stage.  Warp w owns rows 16 w .. 16 w + 15 of the
//                    unit, and lane t of a row the unit's 64-block t (the
//                    order of K within a unit is permuted alike for the
//                    weight and X): per unit a lane forms its two rows' 16
//                    dequantized values bf16(fl32(q[c] * m_hat)) once, in
//                    registers, and expands every 8 packed codes through them
//                    with byte permutes; warp MMAs m16n8k16 with weight rows
//                    as M and tokens as N accumulate in fp32.  When a
//                    CTA leaves a row group it stores its partial tile to the
//                    group's slot for that CTA.  Before streaming, the first
//                    NX CTAs stage their share of the K rows of A and X (bulk
//                    copies) and compute that share of XA = X A (one rank tile
//                    of 8 per warp).
//   k_decode_finish  small CTAs that fit on an SM beside a stream CTA: once
//                    the stream kernel has completed, each adds the NX partial
//                    XA tiles (fixed order) into shared memory, then for its
//                    128 rows the row group's partial tiles in CTA order plus
//                    s (XA B)^T (warp MMAs), and writes Y.
//
// Ordering (programmatic dependent launch).  The stream kernel lets the
// finishing kernel start at once; the finishing kernel waits for the stream
// kernel to complete and then lets the next call start, which it can while
// the finishing kernel still runs: the next stream kernel writes the other
// half of the workspace (calls alternate), reads early only inputs the host
// has checked against this call's writes, and does not complete before its
// predecessor has (every thread waits for it before exiting), so a finishing
// kernel that has waited for its stream kernel has also seen every earlier
// call complete.
//
// Numerics: every weight is the dequantized value bf16(fl32(q[c] * m_hat)) bit
// for bit, and products accumulate in fp32 (the MMA's order).  XA enters the
// LoRA product as a bf16 high part plus a bf16 low part (about 16 significant
// bits).  Results are deterministic (fixed reduction orders).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "convert.cuh"
#include "decode.cuh"
#include "ptx.cuh"

namespace ql {
namespace {

constexpr int CONS = 16;                      // warps of the stream kernel, 16 weight rows each
constexpr int THREADS = CONS * 32;
constexpr int ST_STAGES = 3;                  // ring stages (two with 32 tokens: st_stages<4>)
constexpr int UNIT_ROWS = 256;                // rows per unit
constexpr int UNIT_K = 256;                   // K values per unit (128 packed bytes per row)
constexpr int W_BYTES = UNIT_ROWS * 128;      // packed box of a unit
constexpr int TAB_BYTES = 256 * 256;          // level table (one token tile): 256 entries x 32 lanes x 8 B
constexpr int PD = 2;                         // units of block constants loaded ahead
constexpr int G_MAX = 160;                    // persistent CTAs at most (one per SM)
constexpr int MAX_TOKS = 32;                  // tokens of the largest variant (MT = 4)
constexpr int XA_A_BYTES = 16384;             // staged rows of A per chunk, at most
constexpr int XA_KC_MAX = 256;
constexpr int FIN_WARPS = 4;                  // finishing kernel: 4 warps x 32 rows
constexpr int FIN_ROWS = FIN_WARPS * 32;
// registers of a stream CTA (THREADS threads at the 96-register cap): two never
// fit on one SM (65536 registers), a stream CTA and a finishing CTA do
constexpr int kStreamRegs = THREADS * 96;
static_assert(2 * kStreamRegs > 65536 && kStreamRegs + FIN_WARPS * 32 * 96 <= 65536, "decode CTA residency");

template <int MT>
constexpr int stage_bytes() { return W_BYTES + 4 * (MT * 8) * 128; }
template <int MT>
constexpr int st_stages() { return MT == 4 ? 2 : ST_STAGES; }
// token columns of a partial tile (slot) and of a partial XA tile: 16, or 32 with MT = 4
template <int MT>
constexpr int toks() { return MT == 4 ? 32 : 16; }
template <int MT>
constexpr int slot_floats() { return UNIT_ROWS * toks<MT>(); }
template <int NT>
constexpr int xa_kc() {
  return (XA_A_BYTES / (NT * 8 * 2) < XA_KC_MAX ? XA_A_BYTES / (NT * 8 * 2) : XA_KC_MAX) / 16 * 16;
}
template <int MT, int NT>
constexpr int xa_smem() {  // A chunk, X chunk (toks<MT> rows)
  return xa_kc<NT>() * NT * 8 * 2 + toks<MT>() * xa_kc<NT>() * 2;
}
template <int MT, int NT>
constexpr size_t dec_smem() {
  return (MT == 1 ? TAB_BYTES : 0) + 1024 + (size_t)st_stages<MT>() * stage_bytes<MT>() + (size_t)xa_smem<MT, NT>();
}
// room for a finishing CTA (8 KB of XA, 1 KB reserved) beside a stream CTA in 228 KB
static_assert(dec_smem<2, 16>() + 1024 + 8192 + 1024 <= 228 * 1024, "decode shared memory");
static_assert(dec_smem<2, 1>() + 1024 + 8192 + 1024 <= 228 * 1024, "decode shared memory");
static_assert(dec_smem<4, 16>() + 1024 + 16384 + 1024 <= 228 * 1024, "decode shared memory");

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ uint32_t movtrans(uint32_t v) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(v));
  return r;
}
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
// The dequantized weights of one packed byte's two codes in a row with block
// constant m: bf16(fl32(q[c] * m)) each, from the fp32 level pair at addr
// (element 2j in the low half).
__device__ __forceinline__ uint32_t w_hat_pair(uint32_t addr, float m) {
  const uint2 v = lds64(addr);
  return pack_bf16x2(__fmul_rn(__uint_as_float(v.x), m), __fmul_rn(__uint_as_float(v.y), m));
}
// The 16 dequantized values bf16(fl32(q[c] * m)) of a row-block with block
// constant m, as low-byte (TL) and high-byte (TH) planes: entry c in byte
// c % 4 of word c / 4 (the table lookup8 reads).
__device__ __forceinline__ void w_hat_planes(const float (&q)[16], float m, uint32_t (&TL)[4], uint32_t (&TH)[4]) {
  uint32_t P[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) P[k] = pack_bf16x2(__fmul_rn(q[2 * k], m), __fmul_rn(q[2 * k + 1], m));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    TL[i] = prmt(P[2 * i], P[2 * i + 1], 0x6420u);
    TH[i] = prmt(P[2 * i], P[2 * i + 1], 0x7531u);
  }
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
// One contiguous global -> shared copy completing on `bar` (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}


struct StreamArgs {  // N K / 64 < 2^31 and units < 2^31 (checked on the host)
  int M, K, N;
  int nbox;        // ceil(K / 256)
  int W;           // units = row groups x nbox
  int dq;          // block constants by double quantization (else fp32 absmax)
  int dqt;         // second-level code (QL_DQ_INT8 or QL_DQ_E4M3)
  int w_early;     // the weight may be read before the previous grid completes
  int x_early;     // so may X and A
  int ws_early;    // and this call's workspace half may be written
  int nx;          // CTAs computing partial XA tiles (the first nx)
  int kc;          // rows of A per staged XA chunk
  const int8_t *code;
  const float *step;
  const float *mean;
  const float *absmax;
  const uint16_t *X;   // [M][K]
  const uint16_t *A;   // [K][R]
  float *xap;          // [nx][toks][R] partial XA tiles
  float *slots;        // [groups + G][256 rows][toks tokens]
  int *status;
  float q[16];
};

// CTA that owns unit u when W units are split evenly over G CTAs.
__device__ __forceinline__ int cta_of(int64_t u, int G, int W) { return (int)(((u + 1) * G - 1) / W); }

// ---------------------------------------------------------------------------- XA share
// CTA c < nx takes the K steps of 16 rows [c KS / nx, (c+1) KS / nx),
// KS = K / 16, staged in chunks of kc rows (A rows are contiguous, and so is
// each token's slice of X).  Chunk j is issued by one lane.
template <int NT>
__device__ __forceinline__ void xa_issue(const StreamArgs &a, uint32_t xa_base, uint32_t bar, int j) {
  constexpr int R = NT * 8;
  const int c = blockIdx.x, M = a.M, KC = a.kc, NX = a.nx;
  const int64_t KS = a.K / 16;
  const int64_t k = (int64_t)c * KS / NX * 16 + (int64_t)j * KC, k1 = (int64_t)(c + 1) * KS / NX * 16;
  if (k >= k1) return;
  const int n = (int)min((int64_t)KC, k1 - k);
  const uint32_t xa_a = xa_base, xa_x = xa_base + (uint32_t)(KC * R * 2);
  ptx::fence_proxy_async_smem();  // earlier chunk reads before the copies overwrite them
  ptx::mbar_arrive_expect_tx(bar, (uint32_t)(n * R * 2 + M * n * 2));
  bulk_g2s(xa_a, a.A + k * R, (uint32_t)(n * R * 2), bar);
  for (int m = 0; m < M; ++m)
    bulk_g2s(xa_x + (uint32_t)(m * KC * 2), a.X + (int64_t)m * a.K + k, (uint32_t)(n * 2), bar);
}

// Warp w < NT: rank tile w (columns 8 w .. 8 w + 7) of this CTA's share of XA,
// X as the A fragments (16 tokens per MMA, rows past M zero; with 32 tokens
// two such halves share each A fragment load) and A as the B fragments
// (n = j) through transposing loads; stored (rows < M) to the CTA's partial
// tile.  A chunk after the first is issued once every XA warp has arrived
// at `empty` for the one before.  Returns the number of chunks that landed.
template <int MT, int NT>
__device__ __forceinline__ int xa_share(const StreamArgs &a, uint32_t xa_base, uint32_t bar, uint32_t empty,
                                        volatile int *abort_v) {
  constexpr int R = NT * 8, TH = MT == 4 ? 2 : 1;  // 16-token halves
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int c = blockIdx.x, M = a.M, KC = a.kc, NX = a.nx;
  const int64_t KS = a.K / 16;
  const int64_t k0 = (int64_t)c * KS / NX * 16, k1 = (int64_t)(c + 1) * KS / NX * 16;
  const uint32_t xa_a = xa_base, xa_x = xa_base + (uint32_t)(KC * R * 2);
  float acc[TH][4];
#pragma unroll
  for (int h = 0; h < TH; ++h)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[h][e] = 0.0f;
  int landed_chunks = 0;
#pragma unroll 1
  for (int64_t k = k0; k < k1; k += KC) {
    const int n = (int)min((int64_t)KC, k1 - k);
    if (k > k0 && warp == 0 && lane == 0 &&
        ptx::mbar_wait(empty, (uint32_t)((landed_chunks - 1) & 1), abort_v, a.status))
      xa_issue<NT>(a, xa_base, bar, landed_chunks);
    const bool landed = ptx::mbar_wait(bar, (uint32_t)(landed_chunks & 1), abort_v, a.status);
    if (!__all_sync(0xffffffffu, landed)) return landed_chunks;
    ++landed_chunks;
#pragma unroll 1
    for (int ks = 0; ks < n / 16; ++ks) {
      uint32_t b0, b1;
      ldsm_x2_t(xa_a + (uint32_t)((ks * 16 + (lane & 15)) * R * 2 + warp * 16), b0, b1);
#pragma unroll
      for (int h = 0; h < TH; ++h) {
        const int r0 = 16 * h + g;
        const uint32_t xr = xa_x + (uint32_t)((r0 * KC + ks * 16 + 2 * t) * 2);
        const uint32_t a0 = r0 < M ? lds32(xr) : 0u;
        const uint32_t a2 = r0 < M ? lds32(xr + 16) : 0u;
        const uint32_t a1 = r0 + 8 < M ? lds32(xr + (uint32_t)(8 * KC * 2)) : 0u;
        const uint32_t a3 = r0 + 8 < M ? lds32(xr + (uint32_t)(8 * KC * 2) + 16) : 0u;
        mma16816(acc[h], a0, a1, a2, a3, b0, b1);
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(empty);  // this warp has read the chunk
  }
  if (!a.ws_early) ptx::griddep_wait();  // before the first store to the workspace
  float *mine = a.xap + (int64_t)c * toks<MT>() * R + warp * 8 + 2 * t;
#pragma unroll
  for (int h = 0; h < TH; ++h) {
    const int r0 = 16 * h + g;
    if (r0 < M) __stcg(reinterpret_cast<float2 *>(mine + r0 * R), make_float2(acc[h][0], acc[h][1]));
    if (r0 + 8 < M) __stcg(reinterpret_cast<float2 *>(mine + (r0 + 8) * R), make_float2(acc[h][2], acc[h][3]));
  }
  return landed_chunks;
}

// ---------------------------------------------------------------------------- the weight stream
// At most 96 registers per thread in both kernels, so that a finishing CTA
// (4 warps) fits in the register file beside a stream CTA (16 warps).
template <int MT, int NT>  // MT token tiles of 8, NT rank tiles of 8
__global__ void __maxnreg__(96)
k_decode_stream(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ StreamArgs a) {
  constexpr int XR = MT * 8, SB = stage_bytes<MT>(), ST_STAGES = st_stages<MT>(), TSL = toks<MT>();
  // the finishing kernel may be scheduled now: it waits for this grid to complete
  ptx::griddep_launch();
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint64_t full_bar[ST_STAGES], xa_bar, xa_empty;
  __shared__ unsigned released[ST_STAGES];  // warps done with the stage's current unit
  __shared__ int abort_flag, xa_chunks;
  volatile int *abort_v = &abort_flag;
  // with one token tile the fp32 level table sits at the start
  const uint32_t tab = ptx::smem_u32(smem);
  const uint32_t stages = (tab + (MT == 1 ? TAB_BYTES : 0) + 1023u) & ~1023u;
  const uint32_t xa_base = stages + (uint32_t)(ST_STAGES * SB);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int u0 = (int)((int64_t)c * a.W / G), u1 = (int)((int64_t)(c + 1) * a.W / G);
  const int nu = u1 - u0;
  const int nb_row = a.K >> 6;
  const int rg0 = u0 / a.nbox, b0 = u0 - rg0 * a.nbox;  // first unit's row group and K box
  const bool xa_cta = c < a.nx;
  const int npre = min(nu, ST_STAGES);  // ring stages filled at the start

  // unit i of this CTA (global unit u0 + i) into stage i mod 3
  auto issue = [&](int i, bool w, bool x) {
    const int rg = (u0 + i) / a.nbox, b = (u0 + i) - rg * a.nbox;
    const uint32_t fb = ptx::smem_u32(&full_bar[i % ST_STAGES]), dst = stages + (uint32_t)((i % ST_STAGES) * SB);
    if (w) {
      ptx::mbar_arrive_expect_tx(fb, (uint32_t)SB);
      ptx::tma_load_2d(dst, &tmW, fb, b * 128, rg * UNIT_ROWS);
    }
    if (x)
#pragma unroll
      for (int j = 0; j < 4; ++j) ptx::tma_load_2d(dst + W_BYTES + j * XR * 128, &tmX, fb, b * UNIT_K + 64 * j, 0);
  };

  // Setup.  Once the barriers exist, one lane of warp 0 issues the copies of
  // unit 0 (weight box, and X when X may be read early) and one lane of warp
  // 3 the first XA chunk; units 1 and 2 follow once the lookup table is built,
  // so that unit 0 is not shared out with them in the burst of every CTA's
  // first loads and computing can start sooner.
  if (tid == 0) {
    for (int s = 0; s < ST_STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
      released[s] = 0;
    }
    ptx::mbar_init(ptx::smem_u32(&xa_bar), 1);
    ptx::mbar_init(ptx::smem_u32(&xa_empty), NT);
    ptx::fence_mbar_init();
    abort_flag = 0;
    xa_chunks = 0;
  }
  __syncthreads();
  auto issue_first = [&](int i) {
    if (!a.w_early) ptx::griddep_wait();
    issue(i, true, a.x_early);
    if (!a.x_early) {  // X may still be being written: its boxes follow the wait
      ptx::griddep_wait();
      issue(i, false, true);
    }
  };
  if (lane == 0 && warp == 0) {
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmX);
    issue_first(0);
  }
  if (lane == 0 && warp == ST_STAGES && xa_cta) {
    if (!a.x_early) ptx::griddep_wait();
    xa_issue<NT>(a, xa_base, ptx::smem_u32(&xa_bar), 0);
  }
  if constexpr (MT == 1) {
    // entry e (a packed byte), lane l: the fp32 levels (q[e >> 4], q[e & 15])
    // at byte 256 e + 8 l; the high nibble is element 2j, the lower k of the
    // MMA pair
    float4 *tp = reinterpret_cast<float4 *>(smem);
    for (int i = tid; i < 256 * 16; i += THREADS) {
      const float lo = a.q[(i >> 8) & 15], hi = a.q[(i >> 4) & 15];
      tp[i] = make_float4(lo, hi, lo, hi);
    }
  }
  if (lane == 0 && warp >= 1 && warp < npre) issue_first(warp);
  __syncthreads();
  if (!a.w_early) ptx::griddep_wait();

  if (xa_cta && warp < NT) {
    const int n = xa_share<MT, NT>(a, xa_base, ptx::smem_u32(&xa_bar), ptx::smem_u32(&xa_empty), abort_v);
    if (tid == 0) xa_chunks = n;
  }

  // ---- warp w owns rows 16 w .. 16 w + 15 of the unit's row group.  MMA
  // fragment row g (and g + 8) is weight row pg = 2 (g mod 4) + g / 4 (and
  // pg + 8) of the warp's 16: the 8-byte loads of one 16-lane phase then read
  // rows 0, 2, 4, 6 (or 1, 3, 5, 7), whose two 16-byte chunks land in eight
  // distinct positions under the 128-byte swizzle, so they never conflict.
  const int g = lane >> 2, t = lane & 3;
  const int pg = ((g & 3) << 1) | (g >> 2);
  // Token row of the X fragments: with one token tile, fragment column g >= M
  // reads token g mod M instead of a zero row, so lanes share addresses and a
  // 16-byte load of X takes one shared-memory wavefront (M <= 2) or two
  // (M <= 4) instead of four; the products in those columns are ignored.
  const int xg = MT == 1 ? g % a.M : g;
  const uint32_t lanebase = (uint32_t)lane * 8u;
  const float mu = a.dq ? __ldg(a.mean) : 0.0f;

  // block constants of block t of a unit for the lane's 2 rows (16 w + 8 k + pg),
  // loaded PD units ahead as raw values (the code byte and the step, or the
  // absmax): nothing is computed from them until the unit is reached, so the
  // loads stay in flight until then
  struct Pre {
    float a[2], b[2];
    int c[2];
  };
  int prg = rg0, pb = b0;  // unit of the next load_pre call
  auto load_pre = [&](int i) {
    Pre p;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      p.a[k] = p.b[k] = 0.0f;
      p.c[k] = 0;
    }
    const int rg = prg, kb = pb * 4 + t;
    pb = pb + 1 == a.nbox ? 0 : pb + 1;
    prg += pb == 0;
    if (i >= nu || kb >= nb_row) return p;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int row = rg * UNIT_ROWS + warp * 16 + 8 * k + pg;
      if (row < a.N) {
        const int bi = row * nb_row + kb;
        if (a.dq) {
          p.c[k] = __ldg(a.code + bi);
          p.b[k] = __ldg(a.step + (bi >> 8));
        } else {
          p.a[k] = __ldg(a.absmax + bi);
        }
      }
    }
    return p;
  };
  // two register sets taking units in turn (PD = 2), each reloaded for the
  // unit two ahead as soon as its constants are used (no copies between
  // them, which would wait for the loads)
  static_assert(PD == 2, "two alternating sets of block constants");
  Pre pre_a = load_pre(0), pre_b = load_pre(1);

  float acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[mt][e] = 0.0f;

  // Leave row group rg: store this CTA's partial tile to slot rg + c.
  bool waited = a.ws_early != 0;
  auto flush = [&](int rg) {
    if (!waited) {  // the first store of this warp
      ptx::griddep_wait();
      waited = true;
    }
    float *slot = a.slots + (int64_t)(rg + c) * slot_floats<MT>();
    const int rl = warp * 16 + pg;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      __stcg(reinterpret_cast<float2 *>(slot + rl * TSL + mt * 8 + 2 * t), make_float2(acc[mt][0], acc[mt][1]));
      __stcg(reinterpret_cast<float2 *>(slot + (rl + 8) * TSL + mt * 8 + 2 * t), make_float2(acc[mt][2], acc[mt][3]));
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][e] = 0.0f;
    }
  };

  int cur_rg = -1, rg = rg0, b = b0;
  auto unit = [&](int i, Pre &pre) {
    const int s = i % ST_STAGES;
    if (rg != cur_rg) {
      if (cur_rg >= 0) flush(cur_rg);
      cur_rg = rg;
    }
    // block constants of block t of this unit, rows k = 0, 1
    float mh[2];
#pragma unroll
    for (int k = 0; k < 2; ++k)
      mh[k] = a.dq ? __fadd_rn(__fmul_rn(dq_code_value((int8_t)pre.c[k], a.dqt), pre.b[k]), mu) : pre.a[k];
    pre = load_pre(i + PD);
    // the lane's rows' dequantized values in block t (TL0/TH0: row pg, two or
    // four token tiles only; TL1/TH1: row pg + 8), formed while the stage may
    // still be loading
    uint32_t TL0[4], TH0[4], TL1[4], TH1[4];
    if constexpr (MT > 1) w_hat_planes(a.q, mh[0], TL0, TH0);
    w_hat_planes(a.q, mh[1], TL1, TH1);

    bool landed = false;
    if (!*abort_v)
      landed = ptx::mbar_wait(ptx::smem_u32(&full_bar[s]), (uint32_t)((i / ST_STAGES) & 1), abort_v, a.status);
    const bool ok = __all_sync(0xffffffffu, landed);
    if (ok) {
      const uint32_t wsb = stages + (uint32_t)(s * SB), xsb = wsb + W_BYTES;
      // Step blk: lane t takes K values 16 sg .. 16 sg + 15 of block t, sg =
      // blk ^ t, and its X fragments the same K values (the reduction order
      // is a permutation of the unit's K, the same for both operands).  The
      // packed bytes are 8-byte piece sg of block t's 32 (16-byte chunk
      // 2 t + sg / 2 of the row, at chunk ^ (row mod 8)); X is chunks 2 sg,
      // 2 sg + 1 of block t's 128-byte token row, at chunk ^ (row mod 8).  sg
      // is a Latin square in (t, blk), so no load of a step conflicts on a
      // bank.  Past the row's last block (a ragged unit) the weight and X
      // boxes are zero filled, so those lanes add zero products.
      if constexpr (MT == 4) {
        // 32 tokens: the weights of a step (its 16 A fragments) are formed
        // once and used for two pairs of token tiles in turn, so their cost is
        // shared by all four tiles
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          const int sg = blk ^ t;
          const uint32_t coff = ((uint32_t)((2 * t + (sg >> 1)) ^ pg) << 4) + (uint32_t)(sg & 1) * 8u;
          const uint32_t r0 = wsb + (uint32_t)(warp * 16 + pg) * 128u + coff;
          const uint2 wg = lds64(r0), wg8 = lds64(r0 + 8 * 128);
          uint32_t af[4][4];
          lookup8(wg.x, TL0, TH0, af[0][0], af[0][2], af[1][0], af[1][2]);
          lookup8(wg.y, TL0, TH0, af[2][0], af[2][2], af[3][0], af[3][2]);
          lookup8(wg8.x, TL1, TH1, af[0][1], af[0][3], af[1][1], af[1][3]);
          lookup8(wg8.y, TL1, TH1, af[2][1], af[2][3], af[3][1], af[3][3]);
#pragma unroll
          for (int tp = 0; tp < 2; ++tp) {
            uint32_t xw[2][8];
#pragma unroll
            for (int mm = 0; mm < 2; ++mm) {
              const int mt = 2 * tp + mm;
              const uint32_t rowa = xsb + (uint32_t)(t * XR * 128 + (mt * 8 + g) * 128);
              const uint4 x0 = lds128(rowa + ((uint32_t)((2 * sg) ^ g) << 4));
              const uint4 x1 = lds128(rowa + ((uint32_t)((2 * sg + 1) ^ g) << 4));
              xw[mm][0] = x0.x; xw[mm][1] = x0.y; xw[mm][2] = x0.z; xw[mm][3] = x0.w;
              xw[mm][4] = x1.x; xw[mm][5] = x1.y; xw[mm][6] = x1.z; xw[mm][7] = x1.w;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
              for (int mm = 0; mm < 2; ++mm)
                mma16816(acc[2 * tp + mm], af[j][0], af[j][1], af[j][2], af[j][3], xw[mm][2 * j],
                         xw[mm][2 * j + 1]);
          }
        }
      } else if constexpr (MT == 1) {
        // One token tile: few X loads, so shared memory has room for half of
        // the weights' lookups.  Row pg takes its levels from the shared-memory
        // table (one 64-bit load per packed byte, times the lane's block
        // constant), row pg + 8 from the register planes: the two resources
        // share the work.
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          const int sg = blk ^ t;
          const uint32_t rowa = xsb + (uint32_t)(t * XR * 128 + xg * 128);
          const uint4 x0 = lds128(rowa + ((uint32_t)((2 * sg) ^ xg) << 4));
          const uint4 x1 = lds128(rowa + ((uint32_t)((2 * sg + 1) ^ xg) << 4));
          const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          const uint32_t coff = ((uint32_t)((2 * t + (sg >> 1)) ^ pg) << 4) + (uint32_t)(sg & 1) * 8u;
          const uint32_t r0 = wsb + (uint32_t)(warp * 16 + pg) * 128u + coff;
          const uint2 wg = lds64(r0), wg8 = lds64(r0 + 8 * 128);
          uint32_t af[4][4];
          lookup8(wg8.x, TL1, TH1, af[0][1], af[0][3], af[1][1], af[1][3]);
          lookup8(wg8.y, TL1, TH1, af[2][1], af[2][3], af[3][1], af[3][3]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // MMA j takes K values 16 sg + 4 j + [0, 4): bytes 2j and 2j + 1 of the piece
            const uint32_t wa = (j >> 1) ? wg.y : wg.x;
            const uint32_t s0 = 0x5504u | ((uint32_t)((j & 1) * 2) << 4), s1 = s0 + 0x10u;
            af[j][0] = w_hat_pair(tab + prmt(wa, lanebase, s0), mh[0]);
            af[j][2] = w_hat_pair(tab + prmt(wa, lanebase, s1), mh[0]);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            mma16816(acc[0], af[j][0], af[j][1], af[j][2], af[j][3], xw[2 * j], xw[2 * j + 1]);
        }
      } else {
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          const int sg = blk ^ t;
          uint32_t xw[MT][8];
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t rowa = xsb + (uint32_t)(t * XR * 128 + (mt * 8 + xg) * 128);
            const uint4 x0 = lds128(rowa + ((uint32_t)((2 * sg) ^ xg) << 4));
            const uint4 x1 = lds128(rowa + ((uint32_t)((2 * sg + 1) ^ xg) << 4));
            xw[mt][0] = x0.x; xw[mt][1] = x0.y; xw[mt][2] = x0.z; xw[mt][3] = x0.w;
            xw[mt][4] = x1.x; xw[mt][5] = x1.y; xw[mt][6] = x1.z; xw[mt][7] = x1.w;
          }
          const uint32_t coff = ((uint32_t)((2 * t + (sg >> 1)) ^ pg) << 4) + (uint32_t)(sg & 1) * 8u;
          const uint32_t r0 = wsb + (uint32_t)(warp * 16 + pg) * 128u + coff;
          const uint2 wg = lds64(r0), wg8 = lds64(r0 + 8 * 128);
          // MMA j takes K values 16 sg + 4 j + [0, 4): bytes 2j and 2j + 1 of the piece
          uint32_t af[4][4];
          lookup8(wg.x, TL0, TH0, af[0][0], af[0][2], af[1][0], af[1][2]);
          lookup8(wg.y, TL0, TH0, af[2][0], af[2][2], af[3][0], af[3][2]);
          lookup8(wg8.x, TL1, TH1, af[0][1], af[0][3], af[1][1], af[1][3]);
          lookup8(wg8.y, TL1, TH1, af[2][1], af[2][3], af[3][1], af[3][3]);
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
              mma16816(acc[mt], af[j][0], af[j][1], af[j][2], af[j][3], xw[mt][2 * j], xw[mt][2 * j + 1]);
        }
      }
    }
    // stage s has been read by this warp; the last warp to finish with it
    // loads unit i + 3 into it
    __syncwarp();
    if (lane == 0) {
      unsigned done;
      asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                   : "=r"(done)
                   : "r"(ptx::smem_u32(&released[s]))
                   : "memory");
      if (done == CONS - 1) {
        released[s] = 0;
        if (ok && i + ST_STAGES < nu) {
          ptx::fence_proxy_async_smem();
          issue(i + ST_STAGES, true, true);
        }
      }
    }
    b = b + 1 == a.nbox ? 0 : b + 1;
    rg += b == 0;
  };
#pragma unroll 1
  for (int i = 0; i < nu; i += 2) {
    unit(i, pre_a);
    if (i + 1 < nu) unit(i + 1, pre_b);
  }
  if (cur_rg >= 0) flush(cur_rg);
  // this grid completes only after the grid before it (see the ordering note)
  ptx::griddep_wait();
  // a CTA that gave up lets the copies it still has in flight land before exiting
  __syncthreads();
  if (*abort_v && tid == 0) {
    for (int i = std::max(0, nu - ST_STAGES); i < nu; ++i)
      drain_wait(ptx::smem_u32(&full_bar[i % ST_STAGES]), (uint32_t)((i / ST_STAGES) & 1));
    if (xa_cta) drain_wait(ptx::smem_u32(&xa_bar), (uint32_t)(xa_chunks & 1));
  }
}

// ---------------------------------------------------------------------------- finishing
struct FinArgs {
  int M, N;
  int nbox, W, G;       // the weight stream's unit split
  int nx;               // partial XA tiles
  int x_early;          // B may be read before the stream kernel completes
  int launch_early;     // the stream kernel fills every SM (see k_decode_finish)
  const float *xap;     // [nx][toks][R]
  const float *slots;   // the stream's partial tiles
  const uint16_t *B;    // [R][N]
  float scale;
  uint16_t *Y;          // [M][N]
  uint16_t *XA_out;     // [M][R] bf16 or null
};

template <int MT, int NT>
struct FinShape {
  // k steps, and k steps per chunk of fragments held at once (one with 32
  // tokens, whose XA fragments take four times the registers)
  static constexpr int R = NT * 8, KS = (R + 15) / 16, KSC = MT == 4 ? 1 : (KS < 4 ? KS : 4);
};

// B fragments of k steps [kc0, kc0 + KSC) for the 16 rows from row0 (B is an
// input): 8 x 8 blocks read row-wise, 4 bytes per lane, transposed later.
template <int MT, int NT>
__device__ __forceinline__ void load_bfrag(const FinArgs &a, int row0, int kc0,
                                           uint32_t (&af)[FinShape<MT, NT>::KSC][4]) {
  constexpr int R = FinShape<MT, NT>::R, KSC = FinShape<MT, NT>::KSC;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int kk = 0; kk < KSC; ++kk)
#pragma unroll
    for (int f = 0; f < 4; ++f) {  // a0: (rows 0-7, k 0-7), a1: rows 8-15, a2: k 8-15, a3: both
      const int k = (kc0 + kk) * 16 + 8 * (f >> 1) + g, n = row0 + 8 * (f & 1) + 2 * t;
      af[kk][f] = (k < R && n < a.N) ? __ldg(reinterpret_cast<const uint32_t *>(a.B + (int64_t)k * a.N + n)) : 0u;
    }
}

// XA fragments of k steps [kc0, kc0 + KSC) from shared memory ([M][R] fp32):
// token 8 mt + g, k pairs (16 ks + 2t, +1) and (+8, +9).
template <int MT, int NT>
__device__ __forceinline__ void load_xfrag(const FinArgs &a, const float *xas, int kc0,
                                           float2 (&xf)[FinShape<MT, NT>::KSC][MT][2]) {
  constexpr int R = FinShape<MT, NT>::R, KSC = FinShape<MT, NT>::KSC;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int kk = 0; kk < KSC; ++kk)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int k = (kc0 + kk) * 16 + 2 * t;
      const bool tv = mt * 8 + g < a.M;
      const float *xa = xas + (mt * 8 + g) * R;
      xf[kk][mt][0] = tv && k < R ? *reinterpret_cast<const float2 *>(xa + k) : make_float2(0.0f, 0.0f);
      xf[kk][mt][1] = tv && k + 8 < R ? *reinterpret_cast<const float2 *>(xa + k + 8) : make_float2(0.0f, 0.0f);
    }
}

template <int MT, int NT>
__device__ __forceinline__ void lora_mma(float (&L)[MT][4], const uint32_t (&af)[FinShape<MT, NT>::KSC][4],
                                         const float2 (&xf)[FinShape<MT, NT>::KSC][MT][2]) {
#pragma unroll
  for (int kk = 0; kk < FinShape<MT, NT>::KSC; ++kk) {
    const uint32_t a0 = movtrans(af[kk][0]), a1 = movtrans(af[kk][1]);
    const uint32_t a2 = movtrans(af[kk][2]), a3 = movtrans(af[kk][3]);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const float2 x0 = xf[kk][mt][0], x1 = xf[kk][mt][1];
      const uint32_t h0 = pack_bf16x2(x0.x, x0.y), h1 = pack_bf16x2(x1.x, x1.y);
      const uint32_t l0 = pack_bf16x2(x0.x - bf16lo_to_f32(h0), x0.y - bf16hi_to_f32(h0));
      const uint32_t l1 = pack_bf16x2(x1.x - bf16lo_to_f32(h1), x1.y - bf16hi_to_f32(h1));
      mma16816(L[mt], a0, a1, a2, a3, h0, h1);
      mma16816(L[mt], a0, a1, a2, a3, l0, l1);
    }
  }
}

// Y = bf16(main term + s (XA B)^T): CTA b takes rows 128 b .. 128 b + 127,
// warp w two tiles of 16 of them.
template <int MT, int NT>
__global__ void __maxnreg__(96)
k_decode_finish(const __grid_constant__ FinArgs a) {
  constexpr int R = NT * 8, KS = FinShape<MT, NT>::KS, KSC = FinShape<MT, NT>::KSC, TSL = toks<MT>();
  __shared__ __align__(16) float xas[TSL * R];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int rowc = blockIdx.x * FIN_ROWS + warp * 32;  // this warp's first row
  uint32_t af0[KSC][4];
  if (a.x_early) load_bfrag<MT, NT>(a, rowc, 0, af0);
  // The next call may start once this kernel has waited for the stream kernel
  // (and so for every grid before it).  When the stream kernel has a CTA on
  // every SM it may start at once instead: its CTAs (too large to share an SM
  // with a stream CTA: their registers alone exceed the SM's, see
  // kStreamRegs) then take each SM only when this call's stream CTA on
  // it exits, which that CTA does only after the call before this one has
  // completed; so whatever the next call starts with still sees every call
  // before this one complete, as it would otherwise.
  if (a.launch_early) ptx::griddep_launch();
  ptx::griddep_wait();  // the stream kernel, and every grid before it, completed
  if (!a.launch_early) ptx::griddep_launch();
  if (!a.x_early) load_bfrag<MT, NT>(a, rowc, 0, af0);
  {
    // XA = the partial tiles added in tile order, in two steps: thread t adds
    // tiles zc, zc + zg, ... (zc = t / MR4, zg = 128 / MR4 groups) of element
    // t mod MR4 (4 floats); then the groups' sums are added in group order.
    __shared__ float4 part[FIN_WARPS * 32];
    const int MR4 = a.M * R / 4;
    if (MR4 <= FIN_WARPS * 32) {
      const int zg = (FIN_WARPS * 32) / MR4, i = tid % MR4, zc = tid / MR4;
      float4 sacc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (zc < zg) {
        // a counted loop (the trip count known on entry), so the unrolled
        // loads are issued together rather than one per loop-exit test
        const int cnt = (a.nx - zc + zg - 1) / zg;
        const float4 *src = reinterpret_cast<const float4 *>(a.xap + (int64_t)zc * TSL * R) + i;
        const int64_t step = (int64_t)zg * TSL * R / 4;
#pragma unroll 8
        for (int u = 0; u < cnt; ++u) {
          const float4 v = __ldcg(src + u * step);
          sacc.x += v.x;
          sacc.y += v.y;
          sacc.z += v.z;
          sacc.w += v.w;
        }
      }
      part[tid] = sacc;
      __syncthreads();
      if (tid < MR4) {
        float4 s4 = part[tid];
        for (int q = 1; q < zg; ++q) {
          const float4 v = part[q * MR4 + tid];
          s4.x += v.x;
          s4.y += v.y;
          s4.z += v.z;
          s4.w += v.w;
        }
        reinterpret_cast<float4 *>(xas)[tid] = s4;
      }
    } else {
      for (int i = tid; i < MR4; i += FIN_WARPS * 32) {
        float4 s4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 8
        for (int z = 0; z < a.nx; ++z) {
          const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.xap + (int64_t)z * TSL * R) + i);
          s4.x += v.x;
          s4.y += v.y;
          s4.z += v.z;
          s4.w += v.w;
        }
        reinterpret_cast<float4 *>(xas)[i] = s4;
      }
    }
    __syncthreads();
    if (a.XA_out && blockIdx.x == 0)
      for (int i = tid; i < MR4; i += FIN_WARPS * 32) {
        const float4 s4 = reinterpret_cast<const float4 *>(xas)[i];
        reinterpret_cast<uint32_t *>(a.XA_out)[2 * i] = pack_bf16x2(s4.x, s4.y);
        reinterpret_cast<uint32_t *>(a.XA_out)[2 * i + 1] = pack_bf16x2(s4.z, s4.w);
      }
  }
  __syncthreads();
#pragma unroll 1
  for (int tile = 0; tile < 2; ++tile) {
    const int row0 = rowc + tile * 16;
    if (row0 >= a.N) break;  // N % 8 == 0: rows g of a live tile are valid
    if (tile) load_bfrag<MT, NT>(a, row0, 0, af0);
    const int rg = row0 / UNIT_ROWS;
    const int rowg = row0 + g, rowg8 = rowg + 8;
    const bool vg8 = rowg8 < a.N;
    const int cf = cta_of((int64_t)rg * a.nbox, a.G, a.W), cl = cta_of((int64_t)(rg + 1) * a.nbox - 1, a.G, a.W);
    const int rl = row0 - rg * UNIT_ROWS + g;
    const float *base = a.slots + (int64_t)(rg + cf) * slot_floats<MT>();
    float2 sm[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) sm[mt][0] = sm[mt][1] = make_float2(0.0f, 0.0f);
    constexpr int ZB = MT == 1 ? 8 : (MT == 2 ? 4 : 2);  // partial tiles loaded per batch
#pragma unroll 1
    for (int z0 = 0; z0 <= cl - cf; z0 += ZB) {
      float2 v[ZB][MT][2];
#pragma unroll
      for (int dz = 0; dz < ZB; ++dz)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const bool in = z0 + dz <= cl - cf;
          const float *pz = base + (int64_t)(z0 + dz) * slot_floats<MT>() + mt * 8 + 2 * t;
          v[dz][mt][0] = in ? __ldcg(reinterpret_cast<const float2 *>(pz + rl * TSL)) : make_float2(0.0f, 0.0f);
          v[dz][mt][1] = in ? __ldcg(reinterpret_cast<const float2 *>(pz + (rl + 8) * TSL)) : make_float2(0.0f, 0.0f);
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
    float2 xf[KSC][MT][2];
    load_xfrag<MT, NT>(a, xas, 0, xf);
    lora_mma<MT, NT>(L, af0, xf);
#pragma unroll
    for (int kc0 = KSC; kc0 < KS; kc0 += KSC) {
      uint32_t af[KSC][4];
      load_bfrag<MT, NT>(a, row0, kc0, af);
      load_xfrag<MT, NT>(a, xas, kc0, xf);
      lora_mma<MT, NT>(L, af, xf);
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
  bool attr[3][5] = {};
};
DevInfo &dev_info(int dev) {
  static DevInfo info[64];
  return info[dev & 63];
}

// One half of the workspace: partial XA tiles, then the slots.
struct WsLayout {
  size_t slots, total;
};
WsLayout ws_layout(int64_t N, int r) {
  const size_t groups = (size_t)((N + UNIT_ROWS - 1) / UNIT_ROWS);
  WsLayout l{};
  l.slots = up256((size_t)G_MAX * MAX_TOKS * r * 4);
  l.total = l.slots + (groups + G_MAX) * (size_t)UNIT_ROWS * MAX_TOKS * 4;
  return l;
}

template <typename F>
int max_carveout(F *fn) {
  return check_cuda(cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared),
                    "decode: shared-memory carveout");
}

template <int MT, int NT>
int launch_t(const DecodeProblem &p, StreamArgs &a, FinArgs &f, int G, DevInfo &di, int ti, cudaStream_t st) {
  constexpr int mi = MT == 4 ? 2 : MT - 1;
  if (!di.attr[mi][ti]) {
    int rc = check_cuda(cudaFuncSetAttribute(k_decode_stream<MT, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)dec_smem<MT, NT>()),
                        "decode: shared-memory attribute");
    // both kernels ask for the largest carveout, so a finishing CTA fits beside a stream CTA
    if (!rc) rc = max_carveout(k_decode_stream<MT, NT>);
    if (!rc) rc = max_carveout(k_decode_finish<MT, NT>);
    if (rc) return rc;
    di.attr[mi][ti] = true;
  }
  a.kc = xa_kc<NT>();
  // CTAs computing partial XA tiles: enough that each stages one chunk, at least 32
  const int64_t need = (p.K + a.kc - 1) / a.kc;
  a.nx = (int)std::min<int64_t>(G, std::max<int64_t>(32, need));
  f.nx = a.nx;
  CUtensorMap tmW, tmX;
  int rc = make_tmaps(&tmW, &tmX, p.w.packed, p.N, p.K, p.X, p.M, MT * 8);
  if (rc) return rc;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = dec_smem<MT, NT>();
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_decode_stream<MT, NT>, tmW, tmX, a);
  count_launch();
  rc = check_cuda(e, "decode stream launch");
  if (rc) return rc;
  cudaLaunchConfig_t ff{};
  ff.gridDim = dim3((unsigned)((p.N + FIN_ROWS - 1) / FIN_ROWS));
  ff.blockDim = dim3(FIN_WARPS * 32);
  ff.stream = st;
  ff.attrs = attr;
  ff.numAttrs = 1;
  e = cudaLaunchKernelEx(&ff, k_decode_finish<MT, NT>, f);
  count_launch();
  return check_cuda(e, "decode finish launch");
}

}  // namespace

size_t decode_ws(int64_t N, int64_t K, int r) {
  (void)K;
  return 2 * ws_layout(N, r).total;
}

size_t decode_ws_half(int64_t N, int r) { return ws_layout(N, r).total; }

int launch_decode(const DecodeProblem &p, cudaStream_t st, bool *early_dependents) {
  *early_dependents = false;
  int dev = 0;
  int rc = check_cuda(cudaGetDevice(&dev), "decode: current device");
  if (rc) return rc;
  DevInfo &di = dev_info(dev);
  if (!di.sms) {
    rc = check_cuda(cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev), "decode: SM count");
    if (rc) return rc;
  }
  const int64_t groups = (p.N + UNIT_ROWS - 1) / UNIT_ROWS;
  if (p.N * (p.K / 64) >= ((int64_t)1 << 31) || groups * ((p.K + UNIT_K - 1) / UNIT_K) >= ((int64_t)1 << 31))
    return set_error(QL_ERR_UNSUPPORTED, "decode: %lld x %lld weight too large", (long long)p.N, (long long)p.K);
  const WsLayout l = ws_layout(p.N, p.r);
  char *ws = static_cast<char *>(p.ws) + (p.half ? l.total : 0);
  StreamArgs a{};
  a.M = (int)p.M; a.K = (int)p.K; a.N = (int)p.N;
  a.nbox = (int)((p.K + UNIT_K - 1) / UNIT_K);
  a.W = (int)(groups * a.nbox);
  a.dq = p.w.dq ? 1 : 0;
  a.dqt = p.w.dqt;
  a.w_early = p.w_early ? 1 : 0;
  a.x_early = (p.w_early && p.x_early) ? 1 : 0;
  a.ws_early = p.ws_early ? 1 : 0;
  a.code = p.w.code; a.step = p.w.step; a.mean = p.w.mean; a.absmax = p.w.absmax;
  a.X = p.X; a.A = p.A;
  a.xap = reinterpret_cast<float *>(ws);
  a.slots = reinterpret_cast<float *>(ws + l.slots);
  a.status = device_status_ptr();
  const Codebook &cb = codebook(p.w.qt);
  for (int i = 0; i < 16; ++i) a.q[i] = cb.q[i];
  // every CTA gets at least one unit, so the CTAs of a row group are consecutive
  const int G = (int)std::min<int64_t>(std::min(di.sms, G_MAX), a.W);
  FinArgs f{};
  f.M = a.M; f.N = a.N; f.nbox = a.nbox; f.W = a.W; f.G = G;
  f.x_early = a.x_early;
  f.launch_early = G == di.sms;
  *early_dependents = f.launch_early;
  f.xap = a.xap; f.slots = a.slots;
  f.B = p.B; f.scale = p.scale; f.Y = p.Y; f.XA_out = p.XA_out;
  const int mt = p.M <= 8 ? 1 : (p.M <= 16 ? 2 : 4);  // token tiles of 8
  switch (p.r * 8 + mt) {
#define QL_DEC(R_, TI_)                                                 \
  case R_ * 8 + 1: return launch_t<1, R_ / 8>(p, a, f, G, di, TI_, st); \
  case R_ * 8 + 2: return launch_t<2, R_ / 8>(p, a, f, G, di, TI_, st); \
  case R_ * 8 + 4: return launch_t<4, R_ / 8>(p, a, f, G, di, TI_, st);
    QL_DEC(8, 0) QL_DEC(16, 1) QL_DEC(32, 2) QL_DEC(64, 3) QL_DEC(128, 4)
#undef QL_DEC
    default: return set_error(QL_ERR_UNSUPPORTED, "decode: rank %d", p.r);
  }
}

}  // namespace ql
